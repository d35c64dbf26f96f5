"""The oracle's thread count (used only to time it single-threaded and on all
cores) changes no result: every output element is one thread's ordered sum."""
import numpy as np

import workloads as wl
from oracle import oracle as orc


def test_results_do_not_depend_on_thread_count():
    g = wl.rng(77)
    H, F, E = 96, 64, 5
    experts = [tuple(orc.Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in wl.expert(g, H, F, 4, 32))
               for _ in range(E)]
    x = wl.activations(g, 3, H)
    ids, w = wl.routing_topk_softmax(g, 3, E, 2)
    m = wl.random_matrix(g, 4, 70, H, 32)
    prev = orc.set_threads(1)
    try:
        assert orc.threads() == 1
        y1 = orc.moe_block(H, F, experts, x, ids, w)
        z1 = orc.matmul(m.fmt, m.gs, m.O, m.I, m.data, m.scales, x)
    finally:
        orc.set_threads(prev)
    assert orc.threads() == prev
    yn = orc.moe_block(H, F, experts, x, ids, w)
    zn = orc.matmul(m.fmt, m.gs, m.O, m.I, m.data, m.scales, x)
    assert np.array_equal(y1, yn)
    assert np.array_equal(z1, zn)

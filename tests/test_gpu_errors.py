"""Loud refusals and device-side error reporting on the GPU (no fault is
caused: bad ids are caught by the kernels' own checks and reported through
the error word; injected failures are host-side)."""
import numpy as np
import pytest

import workloads as wl
from gpu_util import cuda_or_skip, upload

pytestmark = pytest.mark.gpu


def _small_table(coli, g, H=128, F=64, E=4, fmt=4, gs=64):
    return coli.ExpertTable([tuple(upload(coli, m) for m in wl.expert(g, H, F, fmt, gs)) for _ in range(E)])


@pytest.mark.parametrize("S", [1, 20])
@pytest.mark.parametrize("fmt,gs", [(4, 64), (5, 64)])
def test_bad_routing_id_is_reported(S, fmt, gs):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(1)
    table = _small_table(coli, g, fmt=fmt, gs=gs)
    ids = np.zeros((S, 2), np.int32)
    ids[-1, 1] = 9    # out of range for 4 experts
    x = torch.zeros(S, 128, device="cuda")
    y = torch.zeros(S, 128, device="cuda")
    coli.moe_block(x, table, torch.from_numpy(ids).cuda(), torch.ones(S, 2, device="cuda"), y)
    with pytest.raises(coli.ColiError) as ei:
        coli.sync_check()
    assert ei.value.code == coli.COLI_EINVAL
    coli.sync_check()   # the error word was cleared


def test_mixed_formats_refused():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(2)
    a = wl.expert(g, 128, 64, 4, 64)
    b = wl.expert(g, 128, 64, 2, 0)
    table = coli.ExpertTable([tuple(upload(coli, m) for m in a), tuple(upload(coli, m) for m in b)])
    with pytest.raises(coli.ColiError) as ei:
        coli.moe_block(torch.zeros(1, 128, device="cuda"), table, torch.zeros(1, 2, dtype=torch.int32, device="cuda"),
                       torch.ones(1, 2, device="cuda"), torch.zeros(1, 128, device="cuda"))
    assert ei.value.code == coli.COLI_EFMT


def test_shape_mismatch_refused():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(3)
    G, U, _ = wl.expert(g, 128, 64, 4, 64)
    D = wl.random_matrix(g, 4, 64, 128, 64)      # transposed: wrong shape
    table = coli.ExpertTable([(upload(coli, G), upload(coli, U), upload(coli, D))])
    with pytest.raises(coli.ColiError) as ei:
        coli.moe_block(torch.zeros(1, 128, device="cuda"), table, torch.zeros(1, 1, dtype=torch.int32, device="cuda"),
                       torch.ones(1, 1, device="cuda"), torch.zeros(1, 128, device="cuda"))
    assert ei.value.code == coli.COLI_EINVAL


def test_fail_after_injects_and_launches_nothing():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(4)
    m = wl.random_matrix(g, 2, 64, 256)
    W = upload(coli, m)
    x = torch.randn(1, 256, device="cuda")
    y = torch.zeros(1, 64, device="cuda")
    coli.set_fail_after(1)
    try:
        coli.matmul(W, x, y)
        before = coli.stats()["launches"]
        y.fill_(123.0)
        with pytest.raises(coli.ColiError) as ei:
            coli.matmul(W, x, y)
        assert ei.value.code == coli.COLI_EINJECTED
        torch.cuda.synchronize()
        assert coli.stats()["launches"] == before
        assert float(y[0, 0]) == 123.0
    finally:
        coli.set_fail_after(-1)
    coli.matmul(W, x, y)
    coli.sync_check()


def test_engagement_counter_counts_launches():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(5)
    W = upload(coli, wl.random_matrix(g, 4, 64, 256, 64))
    x = torch.randn(2, 256, device="cuda")
    y = torch.zeros(2, 64, device="cuda")
    s0 = coli.stats()
    coli.matmul(W, x, y)
    coli.sync_check()
    s1 = coli.stats()
    assert s1["launches"] == s0["launches"] + 1
    assert s1["weight_bytes"] - s0["weight_bytes"] == W.info()["alg_bytes"]

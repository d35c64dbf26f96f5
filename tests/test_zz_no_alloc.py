"""coli_moe_block_noalloc: the decode expert block for callers that cannot
allocate device memory (allocation-free decode loops, memory owned by another
allocator).  Checked through the C ABI against the oracle and against the
allocating entry point coli_moe_block on the same inputs, within the parity
tolerance, on two calls in a row; this file runs last."""
import numpy as np
import pytest

import workloads as wl
from gpu_util import TOL, cuda_or_skip, norm_err, upload
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _setup(coli, g, H, F, E, fmt, gs):
    host = [wl.expert(g, H, F, fmt, gs) for _ in range(E)]
    return coli.ExpertTable([tuple(upload(coli, m) for m in trip) for trip in host])


@pytest.mark.parametrize("S,K,fmt,gs", [(1, 8, 4, 64), (4, 8, 4, 64), (1, 8, 7, 0), (3, 4, 7, 0)])
def test_noalloc_matches_allocating_entry_point(S, K, fmt, gs):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 1024, 512, 16
    g = wl.rng(700 + S + fmt)
    table = _setup(coli, g, H, F, E, fmt, gs)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        x = torch.from_numpy(wl.activations(g, S, H)).cuda()
        ids_h, w_h = wl.routing_topk_softmax(g, S, E, K)
        ids, w = torch.from_numpy(ids_h).cuda(), torch.from_numpy(w_h).cuda()
        y_ref = torch.empty(S, H, device="cuda")
        coli.moe_block(x, table, ids, w, y_ref)
        coli.sync_check()
        y = torch.full((S, H), float("nan"), device="cuda")
        coli.moe_block_noalloc(x, table, ids, w, y, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error {int(err.item())}"
        assert norm_err(y.cpu().numpy(), y_ref.cpu().numpy()) <= TOL, f"call {call}"


def test_noalloc_with_host_resident_experts():
    """Half of the experts in pinned host memory: the no-allocation block
    equals the allocating one."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E, S, K = 1024, 512, 8, 2, 8
    g = wl.rng(705)
    host = [wl.expert(g, H, F, 4, 64) for _ in range(E)]
    table = coli.ExpertTable([tuple((coli.tensor_upload_host(m.fmt, m.gs, m.O, m.I, m.data, m.scales) if e % 2
                                     else upload(coli, m)) for m in trip) for e, trip in enumerate(host)])
    x = torch.from_numpy(wl.activations(g, S, H)).cuda()
    ids_h, w_h = wl.routing_topk_softmax(g, S, E, K)
    ids, w = torch.from_numpy(ids_h).cuda(), torch.from_numpy(w_h).cuda()
    y_ref = torch.empty(S, H, device="cuda")
    coli.moe_block(x, table, ids, w, y_ref)
    coli.sync_check()
    y = torch.full((S, H), float("nan"), device="cuda")
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    coli.moe_block_noalloc(x, table, ids, w, y, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert norm_err(y.cpu().numpy(), y_ref.cpu().numpy()) <= TOL


def test_noalloc_allocates_nothing_after_first_call():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E, S, K = 512, 256, 8, 1, 4
    g = wl.rng(710)
    table = _setup(coli, g, H, F, E, 2, 0)
    x = torch.from_numpy(wl.activations(g, S, H)).cuda()
    ids_h, w_h = wl.routing_topk_softmax(g, S, E, K)
    ids, w = torch.from_numpy(ids_h).cuda(), torch.from_numpy(w_h).cuda()
    y = torch.empty(S, H, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    coli.moe_block_noalloc(x, table, ids, w, y, err)     # first call: symbol lookup
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        coli.moe_block_noalloc(x, table, ids, w, y, err)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert int(err.item()) == 0


def test_noalloc_limits_are_refused():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(720)
    table = _setup(coli, g, 256, 128, 4, 4, 64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    S, K = 9, 8    # 72 routed slots > 64
    with pytest.raises(coli.ColiError) as ei:
        coli.moe_block_noalloc(torch.zeros(S, 256, device="cuda"), table,
                               torch.zeros(S, K, dtype=torch.int32, device="cuda"), torch.ones(S, K, device="cuda"),
                               torch.zeros(S, 256, device="cuda"), err)
    assert ei.value.code == coli.COLI_EINVAL
    assert "no-allocation" in str(ei.value)


def test_noalloc_reports_bad_routing_id():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(730)
    table = _setup(coli, g, 256, 128, 4, 4, 64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ids = torch.tensor([[0, 7]], dtype=torch.int32, device="cuda")   # 7 >= 4 experts
    coli.moe_block_noalloc(torch.zeros(1, 256, device="cuda"), table, ids, torch.ones(1, 2, device="cuda"),
                           torch.zeros(1, 256, device="cuda"), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 2


@pytest.mark.parametrize("S,K,fmt,gs", [(1, 8, 4, 64), (2, 8, 2, 0), (1, 6, 1, 0), (4, 4, 7, 0), (1, 8, 5, 64)])
def test_noalloc_matches_oracle(S, K, fmt, gs):
    """The no-allocation block against the oracle's expert block, directly;
    the table changes between the two calls (its device copy is refreshed)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 1024, 512, 12
    g = wl.rng(760 + S + K + fmt)
    err = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        host = [wl.expert(g, H, F, fmt, gs) for _ in range(E)]
        table = coli.ExpertTable([tuple(upload(coli, m) for m in trip) for trip in host])
        mats = [tuple(orc.Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in trip) for trip in host]
        x_h = wl.activations(g, S, H)
        ids_h, w_h = wl.routing_topk_softmax(g, S, E, K)
        y = torch.full((S, H), float("nan"), device="cuda")
        coli.moe_block_noalloc(torch.from_numpy(x_h).cuda(), table, torch.from_numpy(ids_h).cuda(),
                               torch.from_numpy(w_h).cuda(), y, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0, f"call {call}: device error {int(err.item())}"
        ref = orc.moe_block(H, F, mats, x_h, ids_h, w_h)
        assert norm_err(y.cpu().numpy(), ref) <= TOL, f"call {call}"


def test_noalloc_is_a_counted_compute_call_with_injection():
    """Counted in coli_get_stats like the other compute calls, stopped by the
    host-side fault injection, and a later success clears the error message."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E, K = 512, 256, 4, 2
    g = wl.rng(790)
    table = _setup(coli, g, H, F, E, 4, 64)
    x = torch.from_numpy(wl.activations(g, 1, H)).cuda()
    ids_h, w_h = wl.routing_topk_softmax(g, 1, E, K)
    ids, w = torch.from_numpy(ids_h).cuda(), torch.from_numpy(w_h).cuda()
    y = torch.empty(1, H, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    coli.reset_stats()
    coli.moe_block_noalloc(x, table, ids, w, y, err)
    torch.cuda.synchronize()
    st = coli.stats()
    assert st["calls"] == 1 and st["launches"] >= 1
    coli.set_fail_after(0)
    try:
        with pytest.raises(coli.ColiError) as ex:
            coli.moe_block_noalloc(x, table, ids, w, y, err)
        assert ex.value.code == coli.COLI_EINJECTED
    finally:
        coli.set_fail_after(-1)
    coli.moe_block_noalloc(x, table, ids, w, y, err)
    torch.cuda.synchronize()
    assert coli.last_error() == ""

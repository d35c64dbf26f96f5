"""Host-resident weights (coli_tensor_upload_host): codes and scales stay in
pinned host memory and the kernels read them zero-copy over the CPU-GPU link.
Against the oracle with the same tolerance as device tensors, alone, mixed
with device tensors in one matmul_multi call, and mixed in expert tables."""
import numpy as np
import pytest

import workloads as wl
from gpu_util import TOL, cuda_or_skip, norm_err, upload
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _host(coli, m):
    return coli.tensor_upload_host(m.fmt, m.gs, m.O, m.I, m.data, m.scales)


@pytest.mark.parametrize("fmt,gs", [(0, 0), (1, 0), (2, 0), (3, 0), (4, 64), (4, 6), (5, 16), (7, 0)])
@pytest.mark.parametrize("S", [1, 3, 12])
def test_host_matmul(fmt, gs, S):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(700 + 10 * fmt + S + gs)
    m = wl.random_matrix(g, fmt, 300, 1500, gs)
    x = wl.activations(g, S, 1500)
    W = _host(coli, m)
    assert W.info()["device_bytes"] == 0
    assert W.info()["fmt"] == fmt and W.info()["alg_bytes"] == m.nbytes
    y = torch.full((S, 300), float("nan"), device="cuda")
    coli.matmul(W, torch.from_numpy(x).cuda(), y)
    coli.sync_check()
    assert norm_err(y.cpu().numpy(), orc.matmul(fmt, gs, 300, 1500, m.data, m.scales, x)) <= TOL


def test_host_and_device_in_one_multi_call():
    """Streamed-size device matrices next to a host one: the call stays correct
    (and leaves the bulk-copy kernel for the plain-load one)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(710)
    mats = [wl.random_matrix(g, 4, O, 6144, 64) for O in (2048, 512, 1024)]
    Ws = [upload(coli, mats[0]), _host(coli, mats[1]), upload(coli, mats[2])]
    x = wl.activations(g, 1, 6144)
    ys = [torch.empty(1, m.O, device="cuda") for m in mats]
    coli.matmul_multi(Ws, torch.from_numpy(x).cuda(), ys)
    coli.sync_check()
    for m, y in zip(mats, ys):
        assert norm_err(y.cpu().numpy(), orc.matmul(4, 64, m.O, 6144, m.data, m.scales, x)) <= TOL


@pytest.mark.parametrize("fmt,gs", [(4, 64), (2, 0), (7, 0), (5, 64)])
@pytest.mark.parametrize("S,K", [(1, 8), (3, 4), (20, 8)])
def test_moe_block_mixed_residency(fmt, gs, S, K):
    """An expert table with some experts in host memory and the rest in HBM:
    decode (S = 1, 3) and prefill (S = 20) paths against the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 1024, 512, 10
    g = wl.rng(720 + S + K + fmt)
    host = [wl.expert(g, H, F, fmt, gs) for _ in range(E)]
    on_host = {1, 4, 5, 9}
    dev = [tuple((_host(coli, m) if e in on_host else upload(coli, m)) for m in trip)
           for e, trip in enumerate(host)]
    table = coli.ExpertTable(dev)
    x = wl.activations(g, S, H)
    ids, w = wl.routing_topk_softmax(g, S, E, K)
    y = torch.full((S, H), float("nan"), device="cuda")
    coli.moe_block(torch.from_numpy(x).cuda(), table, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), y)
    coli.sync_check()
    mats = [tuple(orc.Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in trip) for trip in host]
    assert norm_err(y.cpu().numpy(), orc.moe_block(H, F, mats, x, ids, w)) <= TOL


def test_streamed_decode_shape_with_host_expert():
    """The decode shape that takes the bulk-copy kernel when every expert is in
    HBM (6144 x 2048, int4 g64): one host expert moves the call to a plain-load
    kernel and the result still matches the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E, K = 6144, 2048, 8, 8
    g = wl.rng(730)
    host = [wl.expert(g, H, F, 4, 64) for _ in range(2)]
    trips = [host[e % 2] for e in range(E)]
    dev_trip = tuple(upload(coli, m) for m in host[0])
    host_trip = tuple(_host(coli, m) for m in host[1])
    table = coli.ExpertTable([dev_trip if e % 2 == 0 else host_trip for e in range(E)])
    x = wl.activations(g, 1, H)
    ids = np.arange(K, dtype=np.int32).reshape(1, K)
    w = np.full((1, K), 1.0 / K, np.float32)
    y = torch.empty(1, H, device="cuda")
    coli.moe_block(torch.from_numpy(x).cuda(), table, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), y)
    coli.sync_check()
    mats = [tuple(orc.Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in trip) for trip in trips]
    assert norm_err(y.cpu().numpy(), orc.moe_block(H, F, mats, x, ids, w)) <= TOL

"""coli_moe_topk / coli_moe_router on the GPU against the oracle.

The router's decisions (which experts, where top-p cuts) are taken in f32 on
both sides with one rounding per operation, so ids must match exactly and the
weights to the last bit or two (the only difference allowed is the double
exponential inside the sigmoid rounding to f32 differently, which is rare).
"""
import numpy as np
import pytest

import workloads as wl
from gpu_util import TOL, cuda_or_skip, norm_err, upload
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _topk_gpu(coli, torch, logits, K, bias=None, top_p=0.0, norm=False, scale=1.0):
    S, E = logits.shape
    ld = torch.from_numpy(np.ascontiguousarray(logits)).cuda()
    bd = None if bias is None else torch.from_numpy(np.ascontiguousarray(bias)).cuda()
    ids = torch.full((S, K), -7, dtype=torch.int32, device="cuda")
    w = torch.full((S, K), float("nan"), device="cuda")
    coli.moe_topk(ld, K, ids, w, bias=bd, top_p=top_p, norm_topk=norm, routed_scale=scale)
    coli.sync_check()
    return ids.cpu().numpy(), w.cpu().numpy()


def _logits(g, S, E, ties=True):
    l = g.normal(0.0, 1.5, (S, E)).astype(np.float32)
    if ties and E >= 8:
        l[:, 3] = l[:, E - 2]     # exact ties in every row
        l[:, 1] = l[:, 5]
    return l


@pytest.mark.parametrize("S,E,K", [(1, 256, 8), (7, 256, 8), (544, 256, 8), (5, 8, 8), (3, 1000, 64), (9, 37, 1)])
@pytest.mark.parametrize("bias,top_p,norm,scale", [(False, 0.0, False, 1.0), (True, 0.0, True, 2.5),
                                                   (True, 0.6, True, 1.0), (False, 0.9, False, 0.5)])
def test_topk_matches_oracle(S, E, K, bias, top_p, norm, scale):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(9000 + S + E + K + int(bias) + int(10 * top_p))
    l = _logits(g, S, E)
    b = g.normal(0.0, 0.2, E).astype(np.float32) if bias else None
    if b is not None and E >= 8:
        b[3] = b[E - 2]
        b[1] = b[5]
    ids, w = _topk_gpu(coli, torch, l, K, b, top_p, norm, scale)
    rid, rw = orc.moe_topk(l, K, bias=b, top_p=top_p, norm_topk=norm, routed_scale=scale)
    assert np.array_equal(ids, rid)
    assert np.allclose(w, rw, rtol=1e-6, atol=0.0)


def test_topk_saturated_and_equal_logits():
    """Logits that saturate the sigmoid (all keys equal): the picks are the
    lowest ids; a -inf bias pushes an expert last."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    l = np.full((2, 16), 40.0, np.float32)
    l[1] = -40.0
    b = np.zeros(16, np.float32)
    b[0] = -np.inf
    for bias in (None, b):
        ids, w = _topk_gpu(coli, torch, l, 4, bias)
        rid, rw = orc.moe_topk(l, 4, bias=bias)
        assert np.array_equal(ids, rid)
        assert np.array_equal(w, rw)


def test_router_end_to_end_exact():
    """coli_moe_router with an f32 router of small integers and integer x: the
    logits are exact in f32 on both sides, so the routing must match the oracle
    (oracle matmul, then oracle top-K) exactly; the routing then drives
    coli_moe_block."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(9100)
    E, H, F, S, K = 64, 512, 256, 5, 6
    Wr = (g.integers(-3, 4, (E, H)) / 64.0).astype(np.float32)
    x = g.integers(-4, 5, (S, H)).astype(np.float32)
    b = (g.integers(-8, 9, E) / 256.0).astype(np.float32)
    Rt = coli.tensor_upload(0, 0, E, H, Wr, None)
    xd = torch.from_numpy(x).cuda()
    bd = torch.from_numpy(b).cuda()
    ids = torch.empty((S, K), dtype=torch.int32, device="cuda")
    w = torch.empty((S, K), device="cuda")
    coli.moe_router(xd, Rt, K, ids, w, bias=bd, top_p=0.8, norm_topk=True, routed_scale=1.5)
    coli.sync_check()
    logits = orc.matmul(0, 0, E, H, Wr, None, x)
    rid, rw = orc.moe_topk(logits, K, bias=b, top_p=0.8, norm_topk=True, routed_scale=1.5)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(w.cpu().numpy(), rw, rtol=1e-6, atol=0.0)
    # the routing feeds the expert block
    host = [wl.expert(g, H, F, 4, 64) for _ in range(4)]
    host = [host[e % 4] for e in range(E)]
    dev = {}
    table = coli.ExpertTable([dev.setdefault(id(t), tuple(upload(coli, m) for m in t)) for t in host])
    y = torch.full((S, H), float("nan"), device="cuda")
    coli.moe_block(xd, table, ids, w, y)
    coli.sync_check()
    mats = [tuple(orc.Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in t) for t in host]
    ref = orc.moe_block(H, F, mats, x, rid, rw)
    assert norm_err(y.cpu().numpy(), ref) <= TOL


def test_topk_refusals():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    l = torch.zeros((2, 8), device="cuda")
    ids = torch.empty((2, 9), dtype=torch.int32, device="cuda")
    w = torch.empty((2, 9), device="cuda")
    with pytest.raises(coli.ColiError):
        coli.moe_topk(l, 9, ids, w)            # K > n_experts
    with pytest.raises(coli.ColiError):
        coli.moe_topk(l, 0, ids, w)            # K < 1
    with pytest.raises(coli.ColiError):
        coli.moe_topk(l, 2, ids, w, top_p=float("nan"))


def test_router_fp8_weights_exact():
    """A router stored as FP8 (fmt=7, 128x128 block scales) with values that
    make every logit exact in f32 (multiples of 1/4 up to 8, power-of-two block
    scales, integer x): the routing equals the oracle's bit for bit."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(9200)
    E, H, S, K = 256, 6144, 3, 8
    vals = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ok = np.flatnonzero(np.isfinite(vals) & (np.abs(vals) <= 8) & (np.mod(vals * 4, 1) == 0)).astype(np.uint8)
    data = g.choice(ok, (E, H))
    sc = (2.0 ** g.integers(-2, 3, wl.scale_count(7, E, H, 0))).astype(np.float32)
    x = g.integers(-4, 5, (S, H)).astype(np.float32)
    b = (g.integers(-8, 9, E) / 256.0).astype(np.float32)
    Rt = coli.tensor_upload(7, 0, E, H, data, sc)
    ids = torch.empty((S, K), dtype=torch.int32, device="cuda")
    w = torch.empty((S, K), device="cuda")
    coli.moe_router(torch.from_numpy(x).cuda(), Rt, K, ids, w, bias=torch.from_numpy(b).cuda(), norm_topk=True)
    coli.sync_check()
    logits = orc.matmul(7, 0, E, H, data, sc, x)
    rid, rw = orc.moe_topk(logits, K, bias=b, norm_topk=True)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(w.cpu().numpy(), rw, rtol=1e-6, atol=0.0)

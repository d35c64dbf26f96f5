"""coli_moe_block and coli_moe_route on the GPU against the oracle.

Routing indices are compared bit for bit with the oracle's counting sort;
expert-block outputs with max|gpu - oracle| / max|oracle| <= 1e-5.
"""
import numpy as np
import pytest

import workloads as wl
from gpu_util import TOL, cuda_or_skip, norm_err, upload
from oracle import oracle as orc

pytestmark = pytest.mark.gpu


def _experts(g, H, F, E, fmt, gs, distinct=None):
    """E experts; with `distinct`, only that many are drawn and reused."""
    n = E if distinct is None else distinct
    host = [wl.expert(g, H, F, fmt, gs) for _ in range(n)]
    return [host[e % n] for e in range(E)]


def _device_table(coli, host):
    cache = {}
    dev = []
    for trip in host:
        key = id(trip)
        if key not in cache:
            cache[key] = tuple(upload(coli, m) for m in trip)
        dev.append(cache[key])
    return coli.ExpertTable(dev)


def _oracle_mats(host):
    return [tuple(orc.Mat(m.fmt, m.gs, m.O, m.I, m.data, m.scales) for m in trip) for trip in host]


def _run_block(coli, torch, table, x, ids, w, H):
    y = torch.full((x.shape[0], H), float("nan"), device="cuda")
    coli.moe_block(torch.from_numpy(x).cuda(), table, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(), y)
    coli.sync_check()
    return y.cpu().numpy()


@pytest.mark.parametrize("fmt,gs", [(4, 64), (4, 128), (2, 0), (1, 0), (3, 0), (0, 0), (4, 32), (5, 64), (5, 24),
                                    (7, 0)])
@pytest.mark.parametrize("S,K", [(1, 8), (2, 4), (4, 8), (8, 8)])
def test_decode_block(fmt, gs, S, K):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 512, 256, 12
    g = wl.rng(1000 + 7 * fmt + S + K + gs)
    host = _experts(g, H, F, E, fmt, gs)
    x = wl.activations(g, S, H)
    ids, w = wl.routing_topk_softmax(g, S, E, K)
    got = _run_block(coli, torch, _device_table(coli, host), x, ids, w, H)
    ref = orc.moe_block(H, F, _oracle_mats(host), x, ids, w)
    assert norm_err(got, ref) <= TOL


@pytest.mark.parametrize("fmt", [4, 2, 1])
@pytest.mark.parametrize("H,F,gs,K", [(3072, 1536, 64, 8), (6144, 2048, 128, 8), (1024, 512, 64, 3),
                                      (2048, 1024, 32, 16), (1152, 640, 32, 8), (1000, 744, 64, 5),
                                      (6144, 2048, 64, 9)])
def test_decode_streamed_shapes(fmt, H, F, gs, K):
    """S = 1 int4 / int8 shapes taken by the bulk-copy decode kernel: several
    slabs per row, pair ranges that straddle experts and CTAs, partial stages,
    rows whose last 16-byte chunk is partly padding (H, F not multiples of 32),
    the shared expert's ninth slot."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(4100 + H + F + gs + K + 11 * fmt)
    host = _experts(g, H, F, 24, fmt, gs if fmt == 4 else 0, distinct=6)
    x = wl.activations(g, 1, H)
    ids, w = wl.routing_topk_softmax(g, 1, 24, K)
    table = _device_table(coli, host)
    got = _run_block(coli, torch, table, x, ids, w, H)
    ref = orc.moe_block(H, F, _oracle_mats(host), x, ids, w)
    assert norm_err(got, ref) <= TOL
    again = _run_block(coli, torch, table, x, ids, w, H)
    assert np.array_equal(got, again)


def test_decode_streamed_duplicates_and_empty_slots():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F = 1024, 512
    g = wl.rng(4200)
    host = _experts(g, H, F, 8, 4, 64)
    table = _device_table(coli, host)
    mats = _oracle_mats(host)
    x = wl.activations(g, 1, H)
    for ids in (np.array([[3, 3, -1, 5]], np.int32), np.array([[7, 0, 7, 7]], np.int32),
                np.array([[-1, -1, -1, -1]], np.int32)):
        w = g.uniform(0.05, 1.0, ids.shape).astype(np.float32)
        got = _run_block(coli, torch, table, x, ids, w, H)
        ref = orc.moe_block(H, F, mats, x, ids, w)
        if np.all(ids < 0):
            assert np.all(got == 0.0)
        else:
            assert norm_err(got, ref) <= TOL


@pytest.mark.parametrize("K", [4, 9, 16])
def test_int3_decode_duplicates_and_empty_slots(K):
    """int3 decode block: duplicate ids, empty slots, a token with no expert,
    K from 4 to 16."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 1000, 2100, 10
    g = wl.rng(4250 + K)
    host = _experts(g, H, F, E, 5, 40)
    table = _device_table(coli, host)
    mats = _oracle_mats(host)
    x = wl.activations(g, 3, H)
    ids = g.integers(0, E, (3, K)).astype(np.int32)
    ids[0, 1] = ids[0, 0]
    ids[0, K - 1] = -1
    ids[1, :] = -1
    w = g.uniform(0.05, 1.0, ids.shape).astype(np.float32)
    got = _run_block(coli, torch, table, x, ids, w, H)
    ref = orc.moe_block(H, F, mats, x, ids, w)
    assert np.all(got[1] == 0.0)
    assert norm_err(got, ref) <= TOL


def test_int3_decode_full_size():
    """int3 g64 decode block at the decode workload's shape (H 6144, F 2048,
    top-8 of 32 experts) against the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E, K = 6144, 2048, 32, 8
    g = wl.rng(4260)
    host = _experts(g, H, F, E, 5, 64, distinct=8)
    x = wl.activations(g, 1, H)
    ids, w = wl.routing_topk_softmax(g, 1, E, K)
    got = _run_block(coli, torch, _device_table(coli, host), x, ids, w, H)
    ref = orc.moe_block(H, F, _oracle_mats(host), x, ids, w)
    assert norm_err(got, ref) <= TOL


@pytest.mark.parametrize("scale", [1e12, 2.0 ** 30, 1e-12])
def test_decode_streamed_activation_magnitudes(scale):
    """Activations far from unit size: the streamed kernel rescales each lane's
    chunk by a power of two before multiplying, so large and tiny inputs keep
    full f32 precision."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F = 2048, 1024
    g = wl.rng(4300)
    host = _experts(g, H, F, 8, 4, 64)
    x = (wl.activations(g, 1, H) * scale).astype(np.float32)
    ids, w = wl.routing_topk_softmax(g, 1, 8, 4)
    got = _run_block(coli, torch, _device_table(coli, host), x, ids, w, H)
    ref = orc.moe_block(H, F, _oracle_mats(host), x, ids, w)
    assert np.all(np.isfinite(got))
    assert norm_err(got, ref) <= TOL


def test_decode_ragged_routing_and_empty_slots():
    """Empty slots (-1), duplicate ids in a row, a row with no expert, the
    shared expert as one more weight-1 expert on every row."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 384, 200, 7
    g = wl.rng(2024)
    host = _experts(g, H, F, E, 4, 64)
    x = wl.activations(g, 4, H)
    ids = np.array([[0, 3, -1, 6], [2, 2, 5, -1], [-1, -1, -1, -1], [6, 1, 0, 4]], np.int32)
    w = g.uniform(0.05, 1.0, ids.shape).astype(np.float32)
    ids[:, 3] = np.where(ids[:, 3] >= 0, ids[:, 3], -1)
    ids_sh = np.concatenate([ids, np.full((4, 1), 6, np.int32)], axis=1)   # expert 6 as the shared expert
    w_sh = np.concatenate([w, np.ones((4, 1), np.float32)], axis=1)
    table = _device_table(coli, host)
    mats = _oracle_mats(host)
    for I_, W_ in ((ids, w), (ids_sh, w_sh)):
        got = _run_block(coli, torch, table, x, I_, W_, H)
        ref = orc.moe_block(H, F, mats, x, I_, W_)
        assert norm_err(got, ref) <= TOL
    got = _run_block(coli, torch, table, x, ids, w, H)
    assert np.all(got[2] == 0.0)


@pytest.mark.parametrize("fmt,gs", [(4, 128), (4, 64), (2, 0), (4, 16), (1, 0), (7, 0), (0, 0), (3, 0), (5, 64)])
@pytest.mark.parametrize("S,K", [(9, 8), (40, 4), (100, 8)])
def test_prefill_block(fmt, gs, S, K):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 384, 160, 24
    g = wl.rng(3000 + S + K + fmt + gs)
    host = _experts(g, H, F, E, fmt, gs)
    x = wl.activations(g, S, H, bf16_exact=True)
    ids, w = wl.routing_zipf(g, S, E, K)
    ids[3, 1] = -1
    got = _run_block(coli, torch, _device_table(coli, host), x, ids, w, H)
    ref = orc.moe_block(H, F, _oracle_mats(host), x, ids, w)
    assert norm_err(got, ref) <= TOL


def test_decode_is_bitwise_deterministic():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 1024, 512, 16
    g = wl.rng(44)
    host = _experts(g, H, F, E, 4, 64)
    table = _device_table(coli, host)
    x = wl.activations(g, 2, H)
    ids, w = wl.routing_topk_softmax(g, 2, E, 8)
    a = _run_block(coli, torch, table, x, ids, w, H)
    b = _run_block(coli, torch, table, x, ids, w, H)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("S,K,E", [(1, 8, 256), (4, 8, 256), (544, 8, 256), (37, 3, 5), (1000, 6, 8192)])
def test_route_bit_exact(S, K, E):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(S + K + E)
    ids = g.integers(-1, E, (S, K)).astype(np.int32)
    off_ref, ord_ref = orc.route(ids, E)
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    order = torch.full((S * K,), -7, dtype=torch.int32, device="cuda")
    coli.moe_route(torch.from_numpy(ids).cuda(), E, off, order)
    coli.sync_check()
    off = off.cpu().numpy()
    assert np.array_equal(off, off_ref)
    assert np.array_equal(order.cpu().numpy()[: len(ord_ref)], ord_ref)


def test_decode_workload_full_size():
    """Decode expert block at full size: H=6144, F=2048, 256 experts, top-8
    softmax routing, fmt=4 gs=64, S=1 (32 distinct seeded experts, each
    resident at 8 addresses)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    c = wl.MOE_DECODE
    g = wl.rng(c["seed"])
    host = _experts(g, c["H"], c["F"], c["E"], c["fmt"], c["gs"], distinct=32)
    table = _device_table(coli, host)
    mats = _oracle_mats(host)
    for rep in range(2):
        x = wl.activations(g, 1, c["H"])
        ids, w = wl.routing_topk_softmax(g, 1, c["E"], c["K"])
        got = _run_block(coli, torch, table, x, ids, w, c["H"])
        ref = orc.moe_block(c["H"], c["F"], mats, x, ids, w)
        assert norm_err(got, ref) <= TOL


def test_prefill_workload_sampled_rows():
    """Prefill expert block at full size (S=544, Zipf(1.1) routing over 256
    experts, fmt=4 gs=128, bf16-representable x); 6 sampled rows checked
    against the oracle (each row depends only on its own x and routing)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    c = wl.MOE_PREFILL
    g = wl.rng(c["seed"])
    host = _experts(g, c["H"], c["F"], c["E"], c["fmt"], c["gs"], distinct=32)
    table = _device_table(coli, host)
    x = wl.activations(g, c["S"], c["H"], bf16_exact=True)
    ids, w = wl.routing_zipf(g, c["S"], c["E"], c["K"], c["zipf"])
    got = _run_block(coli, torch, table, x, ids, w, c["H"])
    rows = np.sort(g.choice(c["S"], 6, replace=False))
    ref = orc.moe_block(c["H"], c["F"], _oracle_mats(host), x[rows], ids[rows], w[rows])
    assert norm_err(got[rows], ref) <= TOL


def test_prefill_workload_hot_expert_tiles():
    """Prefill expert block at full size (as above): for the three experts
    with the most tokens, the first and the last token of every 64-token tile
    of the expert's rows (tokens in routing order, the order the grouped GEMMs
    take them in) checked against the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    c = wl.MOE_PREFILL
    g = wl.rng(c["seed"] + 1)
    host = _experts(g, c["H"], c["F"], c["E"], c["fmt"], c["gs"], distinct=32)
    table = _device_table(coli, host)
    x = wl.activations(g, c["S"], c["H"], bf16_exact=True)
    ids, w = wl.routing_zipf(g, c["S"], c["E"], c["K"], c["zipf"])
    got = _run_block(coli, torch, table, x, ids, w, c["H"])
    counts = np.bincount(ids[ids >= 0].ravel(), minlength=c["E"])
    rows = set()
    for e in np.argsort(-counts, kind="stable")[:3]:
        toks = np.nonzero((ids == e).any(axis=1))[0]   # ascending token order
        for t0 in range(0, len(toks), 64):
            tile = toks[t0: t0 + 64]
            rows.update((int(tile[0]), int(tile[-1])))
    rows = np.array(sorted(rows))
    assert len(rows) >= 6
    ref = orc.moe_block(c["H"], c["F"], _oracle_mats(host), x[rows], ids[rows], w[rows])
    assert norm_err(got[rows], ref) <= TOL


@pytest.mark.parametrize("fmt,gs,S", [(4, 64, 1), (2, 0, 1), (1, 0, 1), (4, 32, 1), (4, 64, 16)])
def test_block_table_handle_matches_array_path(fmt, gs, S):
    """coli_moe_block_t on a table made once runs the same kernels as
    coli_moe_block on the host array: the results agree bit for bit."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E, K = 1024, 512, 16, 8
    g = wl.rng(5100 + fmt + gs + S)
    host = _experts(g, H, F, E, fmt, gs, distinct=8)
    table = _device_table(coli, host)
    x = torch.from_numpy(wl.activations(g, S, H)).cuda()
    ids, w = wl.routing_topk_softmax(g, S, E, K)
    di, dw = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    y1 = torch.full((S, H), float("nan"), device="cuda")
    y2 = torch.full((S, H), float("nan"), device="cuda")
    coli.moe_block(x, table, di, dw, y1)
    coli.moe_block_array(x, table, di, dw, y2)
    coli.sync_check()
    assert torch.equal(y1, y2)
    ref = orc.moe_block(H, F, _oracle_mats(host), x.cpu().numpy(), ids, w)
    assert norm_err(y1.cpu().numpy(), ref) <= TOL


def test_block_table_handle_keeps_one_plan_per_K():
    """One table, calls with K = 4, 8, 4: the table's kept decode plan is the
    one of the call's K each time."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 2048, 1024, 24
    g = wl.rng(5200)
    host = _experts(g, H, F, E, 4, 64, distinct=6)
    table = _device_table(coli, host)
    mats = _oracle_mats(host)
    for K in (4, 8, 4):
        x = wl.activations(g, 1, H)
        ids, w = wl.routing_topk_softmax(g, 1, E, K)
        got = _run_block(coli, torch, table, x, ids, w, H)
        assert norm_err(got, orc.moe_block(H, F, mats, x, ids, w)) <= TOL


@pytest.mark.parametrize("fmt,gs,H,F", [(4, 64, 512, 256), (4, 128, 1024, 512), (2, 0, 384, 192), (4, 64, 2048, 2048),
                                        (4, 128, 4096, 1024)])
@pytest.mark.parametrize("S,K,E", [(40, 4, 24), (20, 2, 24), (60, 2, 2), (33, 8, 64), (100, 8, 64)])
def test_prefill_small_expert_groups(fmt, gs, H, F, S, K, E):
    """Prefill shapes the small-row path takes: experts with at most 12 rows go
    in groups of up to 4 rows to the mma.sync products, the rest to the tensor-
    core GEMMs (mixed; every expert small; no expert small), against the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(5300 + fmt + gs + H + S + K + E)
    host = _experts(g, H, F, E, fmt, gs, distinct=min(E, 8))
    x = wl.activations(g, S, H, bf16_exact=True)
    ids, w = wl.routing_zipf(g, S, E, K)
    ids[1, 0] = -1
    got = _run_block(coli, torch, _device_table(coli, host), x, ids, w, H)
    ref = orc.moe_block(H, F, _oracle_mats(host), x, ids, w)
    assert norm_err(got, ref) <= TOL


def test_prefill_small_expert_groups_general_x():
    """The small-row path with activations that are not bf16-representable
    (the hi / lo halves carry every bit the tolerance needs)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E, S, K = 1024, 512, 32, 48, 4
    g = wl.rng(5400)
    host = _experts(g, H, F, E, 4, 64, distinct=8)
    x = wl.activations(g, S, H) * np.float32(3.7)
    ids, w = wl.routing_zipf(g, S, E, K)
    got = _run_block(coli, torch, _device_table(coli, host), x, ids, w, H)
    ref = orc.moe_block(H, F, _oracle_mats(host), x, ids, w)
    assert norm_err(got, ref) <= TOL


def test_matvec_and_decode_blocks_interleaved_on_one_stream():
    """The streamed matvec (its claimed-stage counter), the tensor-core decode
    block (its epoch and exit counter) and the int8 streamed decode block share
    one stream's counter words: each leaves them as it found them, so any
    interleaving of calls on one stream, captured in a CUDA graph or not, gives
    the oracle's results."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(6100)
    m = wl.random_matrix(g, 4, 1400, 6144, 64)   # 4.3 MB: the tensor-core streamed matvec
    W = upload(coli, m)
    H, F = 1024, 512
    host4 = _experts(g, H, F, 8, 4, 64)
    host1 = _experts(g, H, F, 8, 1, 0)
    t4, t1 = _device_table(coli, host4), _device_table(coli, host1)
    xm = torch.from_numpy(wl.activations(g, 1, 6144)).cuda()
    xb = torch.from_numpy(wl.activations(g, 1, H)).cuda()
    ids, w = wl.routing_topk_softmax(g, 1, 8, 4)
    di, dw = torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda()
    ref_m = orc.matmul(4, 64, 1400, 6144, m.data, m.scales, xm.cpu().numpy())
    ref4 = orc.moe_block(H, F, _oracle_mats(host4), xb.cpu().numpy(), ids, w)
    ref1 = orc.moe_block(H, F, _oracle_mats(host1), xb.cpu().numpy(), ids, w)
    ym = torch.empty(1, 1400, device="cuda")
    y4 = torch.empty(1, H, device="cuda")
    y1 = torch.empty(1, H, device="cuda")
    st = torch.cuda.Stream()

    def seq():
        for _ in range(3):
            coli.matmul(W, xm, ym, stream=st)
            coli.moe_block(xb, t4, di, dw, y4, stream=st)
            coli.matmul(W, xm, ym, stream=st)
            coli.moe_block(xb, t1, di, dw, y1, stream=st)

    def check():
        assert norm_err(ym.cpu().numpy(), ref_m) <= TOL
        assert norm_err(y4.cpu().numpy(), ref4) <= TOL
        assert norm_err(y1.cpu().numpy(), ref1) <= TOL

    with torch.cuda.stream(st):
        seq()
    torch.cuda.synchronize()
    coli.sync_check(st)
    check()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        seq()
    for y in (ym, y4, y1):
        y.fill_(float("nan"))
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    coli.sync_check(st)
    check()


@pytest.mark.parametrize("S,K", [(1, 8), (20, 4)])
def test_int3_and_int4_experts_in_one_table(S, K):
    """An expert table whose experts are int3 or grouped int4 (one device
    format): decode and prefill against the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    H, F, E = 1024, 512, 8
    g = wl.rng(4270 + S)
    host = [wl.expert(g, H, F, 5 if e % 2 else 4, 64) for e in range(E)]
    x = wl.activations(g, S, H)
    ids, w = wl.routing_topk_softmax(g, S, E, K)
    got = _run_block(coli, torch, _device_table(coli, host), x, ids, w, H)
    ref = orc.moe_block(H, F, _oracle_mats(host), x, ids, w)
    assert norm_err(got, ref) <= TOL

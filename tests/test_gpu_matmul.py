"""coli_matmul / coli_matmul_multi on the GPU against the oracle.

Tolerance: max|gpu - oracle| / max|oracle| <= 1e-5 per output tensor (f32
accumulation on the GPU, f64 in the oracle).  Exact integer cases (power-of-
two scales, small integer activations) must match bit for bit, which pins
the group index, the nibble order and the scale placement independently of
any tolerance.
"""
import numpy as np
import pytest

import workloads as wl
from gpu_util import TOL, cuda_or_skip, norm_err, upload
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

FMT_CASES = [(0, 0), (1, 0), (2, 0), (3, 0), (4, 32), (4, 64), (4, 128), (5, 8), (5, 64), (7, 0)]


def _run(coli, torch, m, x):
    W = upload(coli, m)
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    yd = torch.full((x.shape[0], m.O), float("nan"), device="cuda")
    coli.matmul(W, xd, yd)
    coli.sync_check()
    return yd.cpu().numpy()


@pytest.mark.parametrize("fmt,gs", FMT_CASES)
@pytest.mark.parametrize("S", [1, 2, 3, 4, 5, 8])
def test_matvec_formats(fmt, gs, S):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(100 + 10 * fmt + S)
    m = wl.random_matrix(g, fmt, 333, 2500, gs)
    x = wl.activations(g, S, 2500)
    got = _run(coli, torch, m, x)
    ref = orc.matmul(fmt, gs, 333, 2500, m.data, m.scales, x)
    assert norm_err(got, ref) <= TOL


@pytest.mark.parametrize("fmt,gs", FMT_CASES + [(4, 2), (4, 6), (4, 16), (4, 48), (4, 4096), (5, 24), (5, 4096)])
@pytest.mark.parametrize("O,I", [(1, 1), (3, 7), (5, 31), (17, 33), (9, 65), (64, 1023), (7, 1025), (130, 4097)])
def test_ragged_shapes(fmt, gs, O, I):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(O * 131 + I + fmt)
    m = wl.random_matrix(g, fmt, O, I, gs)
    x = wl.activations(g, 2, I)
    got = _run(coli, torch, m, x)
    ref = orc.matmul(fmt, gs, O, I, m.data, m.scales, x)
    assert norm_err(got, ref) <= TOL


@pytest.mark.parametrize("fmt,gs,O,I", [(1, 0, 70, 3000), (2, 0, 70, 3001), (3, 0, 65, 2999), (4, 64, 66, 3000),
                                        (4, 128, 40, 700), (4, 16, 33, 500), (4, 6, 9, 100), (5, 8, 70, 3001),
                                        (5, 64, 66, 3000), (5, 24, 9, 100)])
@pytest.mark.parametrize("S", [1, 4, 20])
def test_exact_integer_cases(fmt, gs, O, I, S):
    """Power-of-two scales and integer x in [-8, 8]: every product and partial
    sum is exact in f32, so the GPU result must equal the oracle bit for bit."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(7 * O + I + S)
    m = wl.random_matrix(g, fmt, O, I, gs)
    m.scales = (2.0 ** g.integers(-2, 3, m.scales.size)).astype(np.float32)
    x = g.integers(-8, 9, (S, I)).astype(np.float32)
    got = _run(coli, torch, m, x)
    ref = orc.matmul(fmt, gs, O, I, m.data, m.scales, x)
    assert np.array_equal(got, ref)


def test_fmt4_wide_group_equals_fmt2():
    """fmt=4 with gs >= I and the same codes/scales gives fmt=2's result."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(77)
    m2 = wl.random_matrix(g, 2, 200, 1000)
    m4 = wl.Matrix(4, 1024, 200, 1000, m2.data, m2.scales)
    x = wl.activations(g, 3, 1000)
    a = _run(coli, torch, m2, x)
    b = _run(coli, torch, m4, x)
    assert norm_err(a, b) <= TOL


@pytest.mark.parametrize("S", [9, 16, 33, 70])
@pytest.mark.parametrize("fmt,gs", [(0, 0), (1, 0), (2, 0), (3, 0), (4, 64), (4, 10), (5, 16), (7, 0)])
def test_large_s_gemm_path(fmt, gs, S):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(500 + S + fmt)
    m = wl.random_matrix(g, fmt, 150, 700, gs)
    x = wl.activations(g, S, 700)
    got = _run(coli, torch, m, x)
    ref = orc.matmul(fmt, gs, 150, 700, m.data, m.scales, x)
    assert norm_err(got, ref) <= TOL


def _fp8_library(b):
    import torch
    return torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


@pytest.mark.parametrize("S", [1, 3, 9])
def test_fp8_decode_table(S):
    """Every FP8 E4M3 byte through the kernels (I = 1, x = 1, unit scales): y is
    the decode table itself, NaN bytes included, bit for bit (matvec for
    S <= 8, the tiled GEMM for S = 9)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    data = np.arange(256, dtype=np.uint8).reshape(256, 1)
    m = wl.Matrix(7, 0, 256, 1, data, np.ones(wl.scale_count(7, 256, 1, 0), np.float32))
    x = np.ones((S, 1), np.float32)
    got = _run(coli, torch, m, x).astype(np.float64)
    ref = orc.matmul(7, 0, 256, 1, m.data, m.scales, x).astype(np.float64)
    want = np.broadcast_to(_fp8_library(data[:, 0]), (S, 256))
    for a in (ref, want):
        assert np.array_equal(np.isnan(got), np.isnan(a))
        assert np.array_equal(got[~np.isnan(got)], a[~np.isnan(a)])


@pytest.mark.parametrize("O,I", [(300, 3000), (129, 385), (1, 17), (1000, 6144), (777, 6144)])
@pytest.mark.parametrize("S", [1, 4, 20])
def test_fp8_exact_integer_cases(O, I, S):
    """FP8 bytes whose values are multiples of 1/4 up to 8, power-of-two block
    scales and integer x in [-4, 4]: every partial sum is exact in f32, so the
    GPU must equal the oracle bit for bit (block index, partial blocks)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(31 * O + I + S)
    vals = _fp8_library(np.arange(256, dtype=np.uint8))
    ok = np.flatnonzero(np.isfinite(vals) & (np.abs(vals) <= 8) & (np.mod(vals * 4, 1) == 0)).astype(np.uint8)
    data = g.choice(ok, (O, I))
    sc = (2.0 ** g.integers(-2, 3, wl.scale_count(7, O, I, 0))).astype(np.float32)
    m = wl.Matrix(7, 0, O, I, data, sc)
    x = g.integers(-4, 5, (S, I)).astype(np.float32)
    got = _run(coli, torch, m, x)
    ref = orc.matmul(7, 0, O, I, m.data, m.scales, x)
    assert np.array_equal(got, ref)


def test_fp8_matmul_multi():
    """Several FP8 matrices sharing one input (different O, partial blocks)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(92)
    mats = [wl.random_matrix(g, 7, O, 1536) for O in (100, 257, 31, 512)]
    x = wl.activations(g, 2, 1536)
    Ws = [upload(coli, m) for m in mats]
    xd = torch.from_numpy(x).cuda()
    ys = [torch.empty(2, m.O, device="cuda") for m in mats]
    coli.matmul_multi(Ws, xd, ys)
    coli.sync_check()
    for m, y in zip(mats, ys):
        ref = orc.matmul(7, 0, m.O, 1536, m.data, m.scales, x)
        assert norm_err(y.cpu().numpy(), ref) <= TOL


def test_matmul_multi_shared_input():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(91)
    mats = [wl.random_matrix(g, 4, O, 1536, gs) for O, gs in ((100, 64), (257, 128), (31, 32), (512, 64))]
    x = wl.activations(g, 2, 1536)
    Ws = [upload(coli, m) for m in mats]
    xd = torch.from_numpy(x).cuda()
    ys = [torch.empty(2, m.O, device="cuda") for m in mats]
    coli.matmul_multi(Ws, xd, ys)
    coli.sync_check()
    for m, y in zip(mats, ys):
        ref = orc.matmul(4, m.gs, m.O, 1536, m.data, m.scales, x)
        assert norm_err(y.cpu().numpy(), ref) <= TOL


def test_single_gemv_workload():
    """The single grouped-int4 GEMV: S=1, I=2048, O=1536, gs=64."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    c = wl.GEMV_SINGLE
    g = wl.rng(c["seed"])
    m = wl.random_matrix(g, 4, c["O"], c["I"], c["gs"])
    x = wl.activations(g, 1, c["I"])
    got = _run(coli, torch, m, x)
    ref = orc.matmul(4, c["gs"], c["O"], c["I"], m.data, m.scales, x)
    assert norm_err(got, ref) <= TOL


@pytest.mark.parametrize("fmt,gs", [(0, 0), (1, 0), (2, 0), (3, 0), (4, 64), (4, 128), (5, 64)])
@pytest.mark.parametrize("S", [1, 2, 4])
def test_format_sweep_workload(fmt, gs, S):
    """Format sweep at full size: I=6144, O=2048, N(0,0.02) weights quantised
    by symmetric absmax, x ~ N(0,1)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    c = wl.GEMV_SWEEP
    g = wl.rng(c["seed"] + 10 * fmt + gs)
    Wf = g.normal(0.0, 0.02, (c["O"], c["I"])).astype(np.float32)
    m = wl.quantize(fmt, Wf, gs)
    x = wl.activations(g, S, c["I"])
    got = _run(coli, torch, m, x)
    ref = orc.matmul(fmt, gs, c["O"], c["I"], m.data, m.scales, x)
    assert norm_err(got, ref) <= TOL


def test_repeat_is_bitwise_stable():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(5)
    m = wl.random_matrix(g, 4, 777, 3000, 64)
    x = wl.activations(g, 2, 3000)
    a = _run(coli, torch, m, x)
    b = _run(coli, torch, m, x)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("fmt,gs", [(4, 64), (4, 128), (4, 32), (2, 0), (1, 0), (3, 0)])
def test_streamed_matvec_exact_integers(fmt, gs):
    """S = 1 int4 with I a multiple of 128 takes the bulk-copy matvec; with
    power-of-two scales and integer x every step is exact, so the result must
    equal the oracle bit for bit (pins its group index, code placement and the
    removal of the code offset)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(600 + fmt + gs)
    O, I = {1: 700, 3: 2800}.get(fmt, 1404), 6144   # >= 4 MB of weights: the streamed path
    m = wl.random_matrix(g, fmt, O, I, gs)
    m.scales = (2.0 ** g.integers(-2, 3, m.scales.size)).astype(np.float32)
    x = g.integers(-8, 9, (1, I)).astype(np.float32)
    got = _run(coli, torch, m, x)
    ref = orc.matmul(fmt, gs, O, I, m.data, m.scales, x)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt,gs", [(2, 0), (4, 64), (1, 0), (3, 0), (0, 0), (7, 0)])
def test_streamed_matvec_multi(fmt, gs):
    """Eight 2048 x 6144 matrices sharing one input (the weight-streaming
    layer) in one call: rows of all matrices in one index space, CTA row
    blocks that straddle matrices."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(700 + fmt)
    mats = [wl.random_matrix(g, fmt, 2048, 6144, gs) for _ in range(3)]
    mats = [mats[i % 3] for i in range(8)]
    x = wl.activations(g, 1, 6144)
    Ws = [upload(coli, mm) for mm in mats]
    xd = torch.from_numpy(x).cuda()
    ys = [torch.full((1, 2048), float("nan"), device="cuda") for _ in mats]
    coli.matmul_multi(Ws, xd, ys)
    coli.sync_check()
    refs = [orc.matmul(fmt, gs, 2048, 6144, mm.data, mm.scales, x) for mm in mats[:3]]
    for i, y in enumerate(ys):
        assert norm_err(y.cpu().numpy(), refs[i % 3]) <= TOL


@pytest.mark.parametrize("fmt,gs", [(4, 64), (4, 128), (2, 0)])
@pytest.mark.parametrize("S", [2, 3, 4])
def test_streamed_small_s_exact_integers(fmt, gs, S):
    """S = 2..4 int4 with I a multiple of 128 and >= 4 MB of weights takes the
    half-chunk streamed matvec; power-of-two scales and integer x make every
    step exact, so the result must equal the oracle bit for bit."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(800 + fmt + gs + S)
    O, I = 5460, 6144   # > 16 MB of int4 weights: the streamed path for every S
    m = wl.random_matrix(g, fmt, O, I, gs)
    m.scales = (2.0 ** g.integers(-2, 3, m.scales.size)).astype(np.float32)
    x = g.integers(-8, 9, (S, I)).astype(np.float32)
    got = _run(coli, torch, m, x)
    ref = orc.matmul(fmt, gs, O, I, m.data, m.scales, x)
    assert np.array_equal(got, ref)


def _chain_mats(g):
    """A chain of matrices whose shapes compose (x[4096] -> ... -> [4096]) and
    whose launches take different kernels: streamed (int4 groups, int8), the
    register-slab kernel (small int4 matrices) and the generic kernel (FP8)."""
    return [wl.random_matrix(g, 4, 4096, 4096, 64), wl.random_matrix(g, 7, 4096, 4096),
            wl.random_matrix(g, 2, 1024, 4096), wl.random_matrix(g, 4, 4096, 1024, 128),
            wl.random_matrix(g, 1, 4096, 4096)]


def test_dependent_chain_in_graph():
    """Each matvec reads the previous one's output (read after write across
    back-to-back launches, replayed from a CUDA graph): stage k on the GPU
    equals the oracle applied to the GPU's stage k-1 output.  The buffers are
    filled with NaN before every replay, so a stage that read its input
    before the producer finished would not match."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(93)
    mats = _chain_mats(g)
    Ws = [upload(coli, m) for m in mats]
    x = torch.from_numpy(wl.activations(g, 1, 4096)).cuda()
    ys = [torch.empty(1, m.O, device="cuda") for m in mats]
    st = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(st):
        src = x
        for W, y in zip(Ws, ys):
            coli.matmul(W, src, y, stream=st)
            src = y
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=st):
        src = x
        for W, y in zip(Ws, ys):
            coli.matmul(W, src, y, stream=st)
            src = y
    for _ in range(2):
        for y in ys:
            y.fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            graph.replay()
        torch.cuda.synchronize()
        coli.sync_check()
        src = x.cpu().numpy()
        for m, y in zip(mats, ys):
            got = y.cpu().numpy()
            ref = orc.matmul(m.fmt, m.gs, m.O, m.I, m.data, m.scales, src)
            assert norm_err(got, ref) <= TOL
            src = got


def test_ping_pong_chain_in_graph():
    """Two buffers used alternately (each launch overwrites the buffer the
    launch before it read: write after read), replayed from a CUDA graph, against
    the oracle chain in f64 (4 stages, tolerance 4x the per-stage one)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(94)
    mats = [wl.random_matrix(g, 4, 4096, 4096, 64), wl.random_matrix(g, 2, 4096, 4096),
            wl.random_matrix(g, 4, 4096, 4096, 128), wl.random_matrix(g, 1, 4096, 4096)]
    Ws = [upload(coli, m) for m in mats]
    x0 = wl.activations(g, 1, 4096)
    bufs = [torch.empty(1, 4096, device="cuda"), torch.empty(1, 4096, device="cuda")]
    st = torch.cuda.Stream()

    def body():
        for k, W in enumerate(Ws):
            coli.matmul(W, bufs[k % 2], bufs[(k + 1) % 2], stream=st)

    bufs[0].copy_(torch.from_numpy(x0))
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        body()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=st):
        body()
    ref = x0.astype(np.float64)
    for m in mats:
        ref = orc.matmul(m.fmt, m.gs, m.O, m.I, m.data, m.scales, ref.astype(np.float32), want=("y64",))[0]
    for _ in range(3):
        bufs[0].copy_(torch.from_numpy(x0))
        bufs[1].fill_(float("nan"))
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            graph.replay()
        torch.cuda.synchronize()
        coli.sync_check()
        assert norm_err(bufs[0].cpu().numpy(), ref) <= 4 * TOL


@pytest.mark.parametrize("fmt,gs", [(4, 64), (4, 128), (2, 0)])
@pytest.mark.parametrize("O,I", [(4100, 2048), (8200, 1024), (2100, 4096), (1370, 6144)])
@pytest.mark.parametrize("S", [1, 2, 3, 4])
def test_tensor_core_matvec_exact_integers(fmt, gs, O, I, S):
    """S <= 4 int4 with >= 4 MB of weights takes the tensor-core streamed matvec:
    stages of one 16-row tile (rows of more than 2048 inputs) or of two / three
    tiles, warps with fewer segments than the widest, a partial last stage, one
    pair of B columns per row of x.  Power-of-two scales and integer x make
    every step exact: bit-equal to the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(900 + fmt + gs + O + 7 * S)
    m = wl.random_matrix(g, fmt, O, I, gs)
    m.scales = (2.0 ** g.integers(-2, 3, m.scales.size)).astype(np.float32)
    x = g.integers(-8, 9, (S, I)).astype(np.float32)
    got = _run(coli, torch, m, x)
    ref = orc.matmul(fmt, gs, O, I, m.data, m.scales, x)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("fmt,gs", [(4, 64), (2, 0)])
@pytest.mark.parametrize("S", [1, 3])
def test_tensor_core_matvec_multi_ragged(fmt, gs, S):
    """One call over matrices of different heights (stages never straddle two
    matrices; partial stages at every matrix end), random weights and x."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(950 + fmt + S)
    I = 6144
    Os = [2048, 1000, 16, 3, 2047, 640]
    mats = [wl.random_matrix(g, fmt, o, I, gs) for o in Os]
    x = wl.activations(g, S, I)
    Ws = [upload(coli, mm) for mm in mats]
    xd = torch.from_numpy(x).cuda()
    ys = [torch.full((S, o), float("nan"), device="cuda") for o in Os]
    coli.matmul_multi(Ws, xd, ys)
    coli.sync_check()
    for mm, y in zip(mats, ys):
        ref = orc.matmul(fmt, gs, mm.O, I, mm.data, mm.scales, x)
        assert norm_err(y.cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("S", [1, 3, 8, 12])
def test_int3_multi_different_groups(S):
    """coli_matmul_multi over int3 matrices of different O and gs sharing one x
    (the matvec for S <= 8, the tiled GEMM above), each against the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(800 + S)
    I = 9000
    mats = [wl.random_matrix(g, 5, O, I, gs) for O, gs in ((300, 8), (17, 64), (129, 24), (64, 1024))]
    Ws = [upload(coli, m) for m in mats]
    x = wl.activations(g, S, I)
    ys = [torch.full((S, m.O), float("nan"), device="cuda") for m in mats]
    coli.matmul_multi(Ws, torch.from_numpy(x).cuda(), ys)
    coli.sync_check()
    for m, y in zip(mats, ys):
        assert norm_err(y.cpu().numpy(), orc.matmul(5, m.gs, m.O, I, m.data, m.scales, x)) <= TOL


def test_int3_unaligned_activations():
    """int3 matvec with x at a 4-byte (not 16-byte) offset, against the oracle."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(810)
    m = wl.random_matrix(g, 5, 200, 640, 32)
    x = wl.activations(g, 2, 640)
    W = upload(coli, m)
    buf = torch.zeros(2 * 640 + 1, device="cuda")
    buf[1:].copy_(torch.from_numpy(x.reshape(-1)))
    xd = buf[1:].view(2, 640)
    y = torch.full((2, 200), float("nan"), device="cuda")
    coli.matmul(W, xd, y)
    coli.sync_check()
    assert norm_err(y.cpu().numpy(), orc.matmul(5, 32, 200, 640, m.data, m.scales, x)) <= TOL


def test_int3_storage_and_info():
    """An int3 upload reports fmt=5 and its int3 bytes; the device copy holds
    the codes as int4 nibble rows (ceil(I/2) bytes padded to 16) plus the
    scales, and computes the oracle's int3 product on the int4 kernels."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(820)
    O, I, gs = 300, 1000, 40
    m = wl.random_matrix(g, 5, O, I, gs)
    W = upload(coli, m)
    info = W.info()
    assert info["fmt"] == 5 and info["gs"] == gs
    assert info["alg_bytes"] == m.nbytes
    assert info["device_bytes"] == O * (((I + 1) // 2 + 15) // 16 * 16) + 4 * m.scales.size
    x = wl.activations(g, 2, I)
    assert norm_err(_run(coli, torch, m, x), orc.matmul(5, gs, O, I, m.data, m.scales, x)) <= TOL


def test_int3_and_int4_in_one_multi_call():
    """int3 matrices are stored as grouped int4, so one coli_matmul_multi call
    may take both; each result against the oracle in its own format."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(830)
    I = 2048
    mats = [wl.random_matrix(g, 5, 300, I, 64), wl.random_matrix(g, 4, 200, I, 128), wl.random_matrix(g, 5, 77, I, 32)]
    Ws = [upload(coli, m) for m in mats]
    for S in (1, 3, 12):
        x = wl.activations(g, S, I)
        ys = [torch.full((S, m.O), float("nan"), device="cuda") for m in mats]
        coli.matmul_multi(Ws, torch.from_numpy(x).cuda(), ys)
        coli.sync_check()
        for m, y in zip(mats, ys):
            assert norm_err(y.cpu().numpy(), orc.matmul(m.fmt, m.gs, m.O, I, m.data, m.scales, x)) <= TOL

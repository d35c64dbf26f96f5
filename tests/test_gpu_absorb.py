"""kv_b absorption products (coli_matmul_rows / coli_matmul_rows_t) on the GPU
against the oracle: every format, MLA-like head layouts (a row stride larger
than the rows a head uses), ragged shapes, several activation rows, host
resident weights, exact integer cases bit for bit, and argument refusals."""
import numpy as np
import pytest

import workloads as wl
from gpu_util import TOL, cuda_or_skip, norm_err, upload
from oracle import oracle as orc

pytestmark = pytest.mark.gpu

FMTS = [(0, 0), (1, 0), (2, 0), (3, 0), (4, 64), (4, 6), (7, 0), (5, 64)]


def _run(coli, torch, W, m, o0, stride, n_rows, n_heads, x, transposed):
    xd = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    S = x.shape[0]
    out = (S, n_heads, m.I) if transposed else (S, n_heads, n_rows)
    y = torch.full(out, float("nan"), device="cuda")
    (coli.matmul_rows_t if transposed else coli.matmul_rows)(W, o0, stride, n_rows, n_heads, xd, y)
    coli.sync_check()
    return y.cpu().numpy()


def _ref(m, o0, stride, n_rows, n_heads, x, transposed):
    f = orc.matmul_rows_t if transposed else orc.matmul_rows
    return f(m.fmt, m.gs, m.O, m.I, m.data, m.scales, o0, stride, n_rows, n_heads, x)


@pytest.mark.parametrize("fmt,gs", FMTS)
@pytest.mark.parametrize("S", [1, 3, 6])
@pytest.mark.parametrize("transposed", [False, True])
def test_mla_layout(fmt, gs, S, transposed):
    """kv_b of 8 heads x (128 nope + 128 value rows) x 512 latent inputs: the
    key part (rows 0-127 of each head, transposed) and the value part (rows
    128-255, forward)."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(800 + 10 * fmt + S + gs + transposed)
    n_heads, per_head, n_rows, I = 8, 256, 128, 512
    m = wl.random_matrix(g, fmt, n_heads * per_head, I, gs)
    W = upload(coli, m)
    o0 = 0 if transposed else 128
    x = wl.activations(g, S * n_heads, n_rows if transposed else I).reshape(S, n_heads, -1)
    got = _run(coli, torch, W, m, o0, per_head, n_rows, n_heads, x, transposed)
    assert norm_err(got, _ref(m, o0, per_head, n_rows, n_heads, x, transposed)) <= TOL


@pytest.mark.parametrize("fmt,gs", FMTS)
@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("O,I,o0,stride,n_rows,n_heads", [(200, 300, 5, 50, 37, 3), (70, 33, 0, 0, 70, 2),
                                                          (1, 1, 0, 0, 1, 1), (400, 1030, 7, 131, 40, 3)])
def test_ragged(fmt, gs, transposed, O, I, o0, stride, n_rows, n_heads):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(O + I + 7 * fmt + gs + transposed)
    m = wl.random_matrix(g, fmt, O, I, gs)
    W = upload(coli, m)
    x = wl.activations(g, 2 * n_heads, n_rows if transposed else I).reshape(2, n_heads, -1)
    got = _run(coli, torch, W, m, o0, stride, n_rows, n_heads, x, transposed)
    assert norm_err(got, _ref(m, o0, stride, n_rows, n_heads, x, transposed)) <= TOL


@pytest.mark.parametrize("fmt,gs", [(1, 0), (2, 0), (3, 0), (4, 64), (4, 6)])
@pytest.mark.parametrize("transposed", [False, True])
def test_exact_integers(fmt, gs, transposed):
    """Power-of-two scales and integer x in [-8, 8]: every partial sum is exact
    in f32, so the GPU equals the oracle bit for bit."""
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(880 + fmt + gs + transposed)
    O, I, o0, stride, n_rows, n_heads = 520, 512, 4, 128, 96, 4
    m = wl.random_matrix(g, fmt, O, I, gs)
    m.scales = (2.0 ** g.integers(-2, 3, m.scales.size)).astype(np.float32)
    W = upload(coli, m)
    x = g.integers(-8, 9, (5, n_heads, n_rows if transposed else I)).astype(np.float32)
    got = _run(coli, torch, W, m, o0, stride, n_rows, n_heads, x, transposed)
    assert np.array_equal(got, _ref(m, o0, stride, n_rows, n_heads, x, transposed))


@pytest.mark.parametrize("transposed", [False, True])
def test_host_resident(transposed):
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(890 + transposed)
    m = wl.random_matrix(g, 4, 1024, 512, 64)
    W = coli.tensor_upload_host(m.fmt, m.gs, m.O, m.I, m.data, m.scales)
    x = wl.activations(g, 2 * 4, 128 if transposed else 512).reshape(2, 4, -1)
    got = _run(coli, torch, W, m, 0, 256, 128, 4, x, transposed)
    assert norm_err(got, _ref(m, 0, 256, 128, 4, x, transposed)) <= TOL


def test_refusals():
    torch = cuda_or_skip()
    import bit_weight_gemv_fmt1_gb300 as coli
    g = wl.rng(895)
    m = wl.random_matrix(g, 2, 100, 64)
    W = upload(coli, m)
    x = torch.zeros(1, 2, 64, device="cuda")
    y = torch.zeros(1, 2, 64, device="cuda")
    for args in ((0, 60, 50, 2), (-1, 0, 10, 1), (0, 0, 0, 1), (0, 0, 10, 0), (95, 0, 6, 1)):
        with pytest.raises(coli.ColiError):
            coli.matmul_rows(W, *args, x, y)
        with pytest.raises(coli.ColiError):
            coli.matmul_rows_t(W, *args, x, y)

"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself (the pages' worked numbers and byte extremes, closed forms,
library routines on special cases, brute force over raw codes, invariants).

Each pin takes ``mutation`` so the same check runs against the clean oracle
(all must pass) and against builds with one planted mistake (at least one
must fail).  Raw codes are drawn here and packed by ``workloads.pack``; the
expected values are computed from the raw codes with numpy, never from the
packed bytes, so a decoding mistake in the oracle cannot cancel out.
"""
from __future__ import annotations

import math
import os

import numpy as np

import workloads as wl
from oracle import oracle as orc

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _raw(g, fmt, O, I):
    lo, hi = wl.CODE_RANGE[fmt]
    return g.integers(lo, hi + 1, (O, I))


def _deq_from_raw(fmt, gs, codes, scales):
    """Dequantized matrix from raw codes (numpy, f64)."""
    v = codes.astype(np.float64) - wl.OFFSET[fmt]
    O, I = codes.shape
    if fmt in (4, 5):
        ng = wl.n_groups(I, gs)
        s = np.asarray(scales, np.float64).reshape(O, ng)
        return v * np.repeat(s, gs, axis=1)[:, :I]
    return v * np.asarray(scales, np.float64)[:, None]


def pin_golden_layout(mutation=0):
    """tests/golden/nibble_layout.txt: byte extremes and documented element order."""
    for line in open(os.path.join(GOLDEN, "nibble_layout.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        lhs, rhs = line.split("->")
        fmt, hexb = lhs.split()
        fmt = int(fmt)
        want = [int(t) for t in rhs.split()]
        data = np.frombuffer(bytes.fromhex(hexb), dtype=np.uint8).reshape(1, -1)
        I = len(want)
        gs = 2 if fmt == 4 else 0
        sc = np.ones(wl.scale_count(fmt, 1, I, gs), np.float32)
        got = orc.dequant(fmt, gs, 1, I, data, sc, mutation=mutation)[0]
        if list(got) != [float(v) for v in want]:
            return False
    return True


def pin_expert_bytes(mutation=0):
    """Per-expert bytes times the load count round to the printed GB figures."""
    for line in open(os.path.join(GOLDEN, "expert_bytes.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        fmt, gs, H, F, loads, gb = line.split()
        fmt, gs, H, F, loads = int(fmt), int(gs), int(H), int(F), int(loads)
        per = 0
        for (O, I) in ((F, H), (F, H), (H, F)):
            per += O * orc.row_bytes(fmt, I, mutation) + 4 * orc.scale_count(fmt, gs, O, I, mutation)
        if f"{per * loads / 1e9:.3f}" != gb:
            return False
    return True


def pin_all_bytes_brute(mutation=0):
    """All 256 byte values, unit scale: fmt 2/4 and 3 against raw codes."""
    b = np.arange(256, dtype=np.uint8).reshape(1, -1)
    ok = True
    for fmt in (2, 4):
        raw = np.stack([b[0] & 0xF, b[0] >> 4], axis=1).reshape(1, -1).astype(np.int64)
        gs = 512
        got = orc.dequant(fmt, gs, 1, 512, b, np.ones(wl.scale_count(fmt, 1, 512, gs), np.float32),
                          mutation=mutation)
        ok &= np.array_equal(got, raw - 8)
    raw3 = np.stack([(b[0] >> (2 * t)) & 3 for t in range(4)], axis=1).reshape(1, -1).astype(np.int64)
    got3 = orc.dequant(3, 0, 1, 1024, b, np.ones(1, np.float32), mutation=mutation)
    ok &= np.array_equal(got3, raw3 - 2)
    return bool(ok)


def pin_exact_integer_cases(mutation=0):
    """Power-of-two scales and integer x: every product and partial sum is exact
    in f32 and f64, so the oracle's f32 output must equal the integer result."""
    g = wl.rng(11)
    for fmt, gs, O, I in ((1, 0, 7, 33), (2, 0, 5, 31), (3, 0, 6, 45), (4, 16, 5, 70),
                          (4, 64, 4, 200), (4, 6, 3, 29), (4, 128, 3, 77), (5, 8, 5, 37), (5, 64, 4, 200),
                          (5, 24, 3, 50)):
        codes = _raw(g, fmt, O, I)
        sc = (2.0 ** g.integers(-3, 4, wl.scale_count(fmt, O, I, gs))).astype(np.float32)
        x = g.integers(-8, 9, (3, I)).astype(np.float32)
        want = x.astype(np.float64) @ _deq_from_raw(fmt, gs, codes, sc).T
        got = orc.matmul(fmt, gs, O, I, wl.pack(fmt, codes), sc, x, mutation=mutation)
        if not np.array_equal(got.astype(np.float64), want):
            return False
    return True


def pin_random_vs_library(mutation=0):
    """Random codes/scales/x: oracle vs numpy matmul of the matrix dequantized
    from raw codes, within 1e-12 of the sum of |terms| ([T] tolerance form)."""
    g = wl.rng(12)
    for fmt, gs, O, I, S in ((1, 0, 9, 130, 2), (2, 0, 8, 129, 3), (3, 0, 7, 131, 2),
                             (4, 32, 6, 300, 2), (4, 64, 5, 1000, 1), (4, 128, 4, 100, 2),
                             (4, 16, 3, 47, 1), (5, 64, 5, 301, 2), (5, 16, 4, 75, 1)):
        codes = _raw(g, fmt, O, I)
        sc = wl.log_uniform(g, 1e-3, 1e-2, wl.scale_count(fmt, O, I, gs))
        x = g.standard_normal((S, I)).astype(np.float32)
        deq = _deq_from_raw(fmt, gs, codes, sc)
        want = x.astype(np.float64) @ deq.T
        mag = np.abs(x.astype(np.float64)) @ np.abs(deq).T
        y64, = orc.matmul(fmt, gs, O, I, wl.pack(fmt, codes), sc, x, mutation=mutation, want=("y64",))
        if not np.all(np.abs(y64 - want) <= 1e-12 * mag + 1e-300):
            return False
    # fmt=0 is a plain f32 GEMV: numpy in f64
    W = g.normal(0, 0.02, (11, 90)).astype(np.float32)
    x = g.standard_normal((2, 90)).astype(np.float32)
    y64, = orc.matmul(0, 0, 11, 90, W, None, x, mutation=mutation, want=("y64",))
    want = x.astype(np.float64) @ W.astype(np.float64).T
    return bool(np.allclose(y64, want, rtol=0, atol=1e-12))


def pin_int8_unit_scale(mutation=0):
    """fmt=1 with all scales 1 equals an integer matvec (numpy int64)."""
    g = wl.rng(13)
    codes = _raw(g, 1, 10, 64)
    x = g.integers(-100, 101, (2, 64))
    got = orc.matmul(1, 0, 10, 64, wl.pack(1, codes), np.ones(10, np.float32), x.astype(np.float32),
                     mutation=mutation)
    return bool(np.array_equal(got.astype(np.int64), x @ codes.T))


def pin_fmt4_wide_group_is_fmt2(mutation=0):
    """fmt=4 with gs >= I is fmt=2 with a per-row scale (same nibble layout)."""
    g = wl.rng(14)
    for I, gs in ((64, 64), (65, 66), (100, 128), (33, 34)):
        codes = _raw(g, 2, 6, I)
        sc = wl.log_uniform(g, 1e-3, 1e-2, 6)
        x = g.standard_normal((2, I)).astype(np.float32)
        a, = orc.matmul(2, 0, 6, I, wl.pack(2, codes), sc, x, mutation=mutation, want=("y64",))
        b, = orc.matmul(4, gs, 6, I, wl.pack(4, codes), sc, x, mutation=mutation, want=("y64",))
        if not np.array_equal(a, b):
            return False
    return True


def pin_inline_order(mutation=0):
    """Group scale folded in per group equals dequantize-then-multiply, within
    1e-14 of the sum of |terms|."""
    g = wl.rng(15)
    for fmt, gs, O, I in ((4, 64, 6, 500), (4, 16, 4, 97), (2, 0, 5, 99), (1, 0, 5, 77), (3, 0, 4, 70),
                          (7, 0, 260, 300), (5, 32, 5, 203)):
        if fmt == 7:
            m = wl.random_matrix(g, 7, O, I)
            data, sc = m.data, m.scales
        else:
            data = wl.pack(fmt, _raw(g, fmt, O, I))
            sc = wl.log_uniform(g, 1e-3, 1e-2, wl.scale_count(fmt, O, I, gs))
        x = g.standard_normal((2, I)).astype(np.float32)
        y64, mag = orc.matmul(fmt, gs, O, I, data, sc, x, mutation=mutation, want=("y64", "yabs"))
        yi = orc.matmul_inline(fmt, gs, O, I, data, sc, x, mutation=mutation)
        if not np.all(np.abs(y64 - yi) <= 1e-14 * mag):
            return False
    return True


def pin_scale_linearity(mutation=0):
    """y(2s) = 2 y(s) exactly; y(s1+s2) = y(s1) + y(s2) for fmt=4 per group."""
    g = wl.rng(16)
    codes = _raw(g, 4, 5, 200)
    s1 = wl.log_uniform(g, 1e-3, 1e-2, wl.scale_count(4, 5, 200, 64))
    s2 = wl.log_uniform(g, 1e-3, 1e-2, s1.size)
    x = g.standard_normal((2, 200)).astype(np.float32)
    q = wl.pack(4, codes)
    a, = orc.matmul(4, 64, 5, 200, q, s1, x, mutation=mutation, want=("y64",))
    b, = orc.matmul(4, 64, 5, 200, q, (2 * s1).astype(np.float32), x, mutation=mutation, want=("y64",))
    if not np.array_equal(2 * a, b):
        return False
    # additivity with s1 + s2 exactly representable: use powers of two
    p1 = (2.0 ** g.integers(-8, -4, s1.size)).astype(np.float32)
    p2 = (2.0 ** g.integers(-8, -4, s1.size)).astype(np.float32)
    c, = orc.matmul(4, 64, 5, 200, q, p1, x, mutation=mutation, want=("y64",))
    d, m = orc.matmul(4, 64, 5, 200, q, p2, x, mutation=mutation, want=("y64", "yabs"))
    e, = orc.matmul(4, 64, 5, 200, q, (p1 + p2).astype(np.float32), x, mutation=mutation, want=("y64",))
    return bool(np.all(np.abs(c + d - e) <= 1e-13 * m * 4))


def pin_partial_last_group(mutation=0):
    """Glen clamp: with only the last (partial) group's scale non-zero, y is the
    last group's code dot product times that scale."""
    g = wl.rng(17)
    for I, gs in ((100, 64), (70, 16), (129, 32), (10, 4)):
        ng = wl.n_groups(I, gs)
        codes = _raw(g, 4, 3, I)
        sc = np.zeros((3, ng), np.float32)
        sc[:, -1] = 0.5
        x = g.integers(-8, 9, (2, I)).astype(np.float32)
        i0 = (ng - 1) * gs
        want = 0.5 * (x[:, i0:].astype(np.int64) @ (codes[:, i0:] - 8).T)
        got = orc.matmul(4, gs, 3, I, wl.pack(4, codes), sc.reshape(-1), x, mutation=mutation)
        if not np.array_equal(got.astype(np.float64), want.astype(np.float64)):
            return False
    return True


def pin_int3_golden_layout(mutation=0):
    """tests/golden/int3_layout.txt: fmt=5 bytes worked out by hand from the
    layout reading decode to the listed values."""
    for line in open(os.path.join(GOLDEN, "int3_layout.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        lhs, rhs = line.split("->")
        want = [float(t) for t in rhs.split()]
        data = np.frombuffer(bytes.fromhex(lhs.strip()), dtype=np.uint8).reshape(1, -1)
        I = len(want)
        if orc.row_bytes(5, I, mutation) != data.shape[1]:
            return False
        got = orc.dequant(5, 8, 1, I, data, np.ones(wl.n_groups(I, 8), np.float32), mutation=mutation)[0]
        if list(got) != want:
            return False
    return True


def pin_int3_single_codes(mutation=0):
    """fmt=5, brute force over one code at a time: a 3-byte unit holding the
    value v at position t and 0 elsewhere decodes to v - 4 at t and -4
    elsewhere, for all 8 x 8 (t, v); the three bytes are the integer v * 8^t
    written little-endian."""
    for t in range(8):
        for v in range(8):
            data = np.frombuffer((v * 8 ** t).to_bytes(3, "little"), dtype=np.uint8).reshape(1, 3)
            got = orc.dequant(5, 8, 1, 8, data, np.ones(1, np.float32), mutation=mutation)[0]
            want = [-4.0] * 8
            want[t] = float(v - 4)
            if list(got) != want:
                return False
    return True


def pin_int3_within_int4(mutation=0):
    """Every int3 value c - 4 (c = 0..7) is the int4 value of the nibble c + 4,
    and both formats take their group scales the same way, so a fmt=5 matrix
    and the fmt=4 matrix of the same values and scales give the same double
    results (fmt=4 is pinned on its own)."""
    g = wl.rng(23)
    for O, I, gs in ((5, 40, 8), (4, 203, 64), (3, 13, 8), (6, 130, 24), (2, 70, 128)):
        codes = g.integers(0, 8, (O, I))
        sc = wl.log_uniform(g, 1e-3, 1e-2, wl.scale_count(5, O, I, gs))
        x = g.standard_normal((2, I)).astype(np.float32)
        a, = orc.matmul(5, gs, O, I, wl.pack(5, codes), sc, x, mutation=mutation, want=("y64",))
        b, = orc.matmul(4, gs, O, I, wl.pack(4, codes + 4), sc, x, mutation=mutation, want=("y64",))
        if not np.array_equal(a, b):
            return False
    return True


def pin_silu_closed_form(mutation=0):
    """silu(g) = g * sigmoid(g): closed-form values."""
    cases = {0.0: 0.0, 1.0: 1.0 / (1.0 + math.exp(-1.0)), -1.0: -1.0 / (1.0 + math.e),
             2.0: 2.0 / (1.0 + math.exp(-2.0))}
    return all(abs(orc.silu(k, mutation) - v) <= 1e-15 for k, v in cases.items()) and \
        abs(orc.silu(40.0, mutation) - 40.0) < 1e-12 and abs(orc.silu(-40.0, mutation)) < 1e-12


def pin_route_vs_sorted(mutation=0):
    """Counting sort equals Python's stable sorted() over (s, k) slots by id."""
    g = wl.rng(18)
    for S, K, E in ((1, 8, 256), (5, 8, 16), (17, 4, 3), (32, 8, 256)):
        ids = g.integers(-1, E, (S, K)).astype(np.int32)
        offsets, order = orc.route(ids, E, mutation=mutation)
        flat = ids.reshape(-1)
        want = sorted([t for t in range(S * K) if flat[t] >= 0], key=lambda t: flat[t])
        counts = np.bincount(flat[flat >= 0], minlength=E)
        if list(order) != want or not np.array_equal(np.diff(offsets), counts):
            return False
        if offsets[-1] != (flat >= 0).sum():
            return False
    try:
        orc.route(np.array([[0, 3]], np.int32), 3, mutation=mutation)
        return False
    except ValueError:
        return True


def _moe_problem(g, H, F, E, fmt, gs):
    raw = []
    mats = []
    for _ in range(E):
        trip = []
        rtrip = []
        for (O, I) in ((F, H), (F, H), (H, F)):
            c = _raw(g, fmt, O, I)
            sc = wl.log_uniform(g, 1e-2, 5e-2, wl.scale_count(fmt, O, I, gs))
            trip.append(orc.Mat(fmt, gs, O, I, wl.pack(fmt, c), sc))
            rtrip.append(_deq_from_raw(fmt, gs, c, sc))
        mats.append(tuple(trip))
        raw.append(tuple(rtrip))
    return mats, raw


def pin_moe_composition(mutation=0):
    """One expert, w=1, S=1: down(silu(gate x) * (up x)) composed with numpy
    from matrices dequantized from raw codes."""
    g = wl.rng(19)
    H, F = 96, 40
    mats, raw = _moe_problem(g, H, F, 1, 4, 16)
    x = g.standard_normal((1, H)).astype(np.float32)
    y64, = orc.moe_block(H, F, mats, x, np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32),
                         mutation=mutation, want=("y64",))
    G, U, D = raw[0]
    gv = G @ x[0].astype(np.float64)
    uv = U @ x[0].astype(np.float64)
    h = gv / (1.0 + np.exp(-gv)) * uv
    want = D @ h
    mag = np.abs(D) @ np.abs(h)
    return bool(np.all(np.abs(y64[0] - want) <= 1e-12 * mag))


def pin_moe_invariants(mutation=0):
    """Linearity in w, permutation of the expert table, empty slots, the shared
    expert as one more weight-1 expert, duplicate ids counted twice."""
    g = wl.rng(20)
    H, F, E, S, K = 64, 24, 5, 4, 3
    mats, raw = _moe_problem(g, H, F, E, 2, 0)
    x = g.standard_normal((S, H)).astype(np.float32)
    ids = g.integers(0, E, (S, K)).astype(np.int32)
    ids[1, 2] = -1
    ids[2, :] = -1
    w = g.uniform(0.1, 1.0, (S, K)).astype(np.float32)
    y, = orc.moe_block(H, F, mats, x, ids, w, mutation=mutation, want=("y64",))
    y2, = orc.moe_block(H, F, mats, x, ids, (2 * w).astype(np.float32), mutation=mutation, want=("y64",))
    if not np.array_equal(2 * y, y2) or np.any(y[2] != 0):
        return False
    perm = g.permutation(E)
    inv = np.argsort(perm)
    mats_p = [mats[perm[j]] for j in range(E)]
    ids_p = np.where(ids >= 0, inv[np.maximum(ids, 0)], -1).astype(np.int32)
    yp, = orc.moe_block(H, F, mats_p, x, ids_p, w, mutation=mutation, want=("y64",))
    if not np.array_equal(y, yp):
        return False
    # single-slot results against numpy composition (w = 1): catches a dropped weight
    ids1 = np.array([[3]], np.int32)
    y1, = orc.moe_block(H, F, mats, x[:1], ids1, np.full((1, 1), 0.25, np.float32), mutation=mutation,
                        want=("y64",))
    G, U, D = raw[3]
    gv, uv = G @ x[0].astype(np.float64), U @ x[0].astype(np.float64)
    want = 0.25 * (D @ (gv / (1 + np.exp(-gv)) * uv))
    if not np.allclose(y1[0], want, rtol=1e-12, atol=1e-12):
        return False
    # duplicate id counts twice
    yd, = orc.moe_block(H, F, mats, x[:1], np.array([[3, 3]], np.int32),
                        np.full((1, 2), 0.25, np.float32), mutation=mutation, want=("y64",))
    return bool(np.allclose(yd[0], 2 * want, rtol=1e-12, atol=1e-12))


def _sig32(l):
    """sigmoid in double, rounded to f32 (math.exp, element by element)."""
    return np.array([1.0 / (1.0 + math.exp(-float(v))) for v in np.ravel(l)], np.float32).reshape(np.shape(l))


def pin_topk_worked_example(mutation=0):
    """Five logits worked by hand: ties go to the lower id, the bias steers the
    choice but not the weight, top-p keeps the smallest leading set that reaches
    the mass, then norm_topk and routed_scale."""
    l = np.array([[0.0, 1.0, 2.0, 2.0, -1.0]], np.float32)
    sg = _sig32(l[0])
    ids, w = orc.moe_topk(l, 3, mutation=mutation)
    if ids.tolist() != [[2, 3, 1]] or not np.array_equal(w[0], sg[[2, 3, 1]]):
        return False
    ids, w = orc.moe_topk(l, 3, bias=np.array([0, 0, 0, 0, 1], np.float32), mutation=mutation)
    if ids.tolist() != [[4, 2, 3]] or not np.array_equal(w[0], sg[[4, 2, 3]]):
        return False
    # mass of the three: 2*sig(2) + sig(1); half of it is reached after two
    ids, w = orc.moe_topk(l, 3, top_p=0.5, norm_topk=True, routed_scale=2.5, mutation=mutation)
    return ids.tolist() == [[2, 3, -1]] and np.array_equal(w[0], np.array([1.25, 1.25, 0.0], np.float32))


def pin_topk_vs_sort(mutation=0):
    """Greedy argmax equals a stable sort by (-key, id) (brute force), with
    planted ties and a bias; top-p keeps exactly the shortest prefix whose score
    mass reaches top_p of the K scores; norm_topk sums to one."""
    g = wl.rng(77)
    S, E, K = 40, 37, 6
    l = g.normal(0, 1.5, (S, E)).astype(np.float32)
    l[:, 5] = l[:, 9]                      # exact ties in every row
    l[:, 20] = l[:, 11]
    b = g.normal(0, 0.1, E).astype(np.float32)
    b[9] = b[5]
    b[20] = b[11]
    ids, w = orc.moe_topk(l, K, bias=b, mutation=mutation)
    sg = _sig32(l)
    key = (sg + b[None, :]).astype(np.float32)
    for s in range(S):
        order = sorted(range(E), key=lambda e: (-float(key[s, e]), e))[:K]
        if ids[s].tolist() != order or not np.array_equal(w[s], sg[s, order]):
            return False
    ids2, w2 = orc.moe_topk(l, K, bias=b, top_p=0.7, norm_topk=True, mutation=mutation)
    for s in range(S):
        sc = sg[s, ids[s]].astype(np.float64)
        kept = int((ids2[s] >= 0).sum())
        if kept < 1 or ids2[s, :kept].tolist() != ids[s, :kept].tolist() or np.any(ids2[s, kept:] != -1):
            return False
        total = sc.sum()
        if sc[:kept].sum() < 0.7 * total * (1 - 1e-6) or sc[:kept - 1].sum() >= 0.7 * total * (1 + 1e-6):
            return False
        if abs(float(w2[s, :kept].astype(np.float64).sum()) - 1.0) > 1e-6 or np.any(w2[s, kept:] != 0):
            return False
    return True


def _e4m3_library(b):
    """FP8 E4M3 bytes decoded by PyTorch's float8_e4m3fn dtype (f64)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_fp8_block_count(mutation=0):
    """tests/golden/fp8_blocks.txt: the scale count the pages print for fmt=7,
    and one byte per element."""
    for line in open(os.path.join(GOLDEN, "fp8_blocks.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        lhs, rhs = line.split("->")
        O, I = (int(t) for t in lhs.split())
        if orc.scale_count(7, 0, O, I, mutation) != int(rhs) or orc.row_bytes(7, I, mutation) != I:
            return False
    return True


def pin_fp8_all_bytes(mutation=0):
    """All 256 E4M3 bytes at unit scale against PyTorch's float8_e4m3fn
    conversion (NaN at the same two bytes), plus the format's closed-form
    landmarks: largest finite 448 (0x7E), smallest subnormal 2^-9 (0x01),
    smallest normal 2^-6 (0x08), 1.0 (0x38), -2 (0xC0)."""
    b = np.arange(256, dtype=np.uint8).reshape(1, -1)
    got = orc.dequant(7, 0, 1, 256, b, np.ones(2, np.float32), mutation=mutation)[0]
    want = _e4m3_library(b[0])
    if not np.array_equal(np.isnan(got), np.isnan(want)) or not np.array_equal(got[~np.isnan(got)],
                                                                               want[~np.isnan(want)]):
        return False
    marks = {0x7E: 448.0, 0x01: 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0xC0: -2.0, 0x00: 0.0}
    return all(got[k] == v for k, v in marks.items()) and bool(np.isnan(got[0x7F]) and np.isnan(got[0xFF]))


def pin_fp8_block_structure(mutation=0):
    """Brute force over the blocks of a 300 x 130 fmt=7 tensor (3 x 2 blocks,
    partial at the bottom and right): with only block (bo, bi)'s scale set to
    0.5, the dequantized matrix is 0.5 * the library-decoded bytes inside that
    block and zero everywhere else."""
    g = wl.rng(18)
    O, I = 300, 130
    m = wl.random_matrix(g, 7, O, I)
    dec = _e4m3_library(m.data)
    nbo, nbi = wl.n_groups(O, 128), wl.n_groups(I, 128)
    for bo in range(nbo):
        for bi in range(nbi):
            sc = np.zeros(nbo * nbi, np.float32)
            sc[bo * nbi + bi] = 0.5
            got = orc.dequant(7, 0, O, I, m.data, sc, mutation=mutation)
            want = np.zeros((O, I))
            want[bo * 128:(bo + 1) * 128, bi * 128:(bi + 1) * 128] = 0.5 * dec[bo * 128:(bo + 1) * 128,
                                                                               bi * 128:(bi + 1) * 128]
            if not np.array_equal(got, want):
                return False
    return True


def pin_fp8_unit_scale_vs_library(mutation=0):
    """fmt=7 with every block scale 1 is a plain matvec of the decoded bytes:
    numpy f64 over the library decode, within 1e-12 of the sum of |terms|;
    scaling every block by 2 doubles y exactly."""
    g = wl.rng(19)
    O, I = 259, 385
    m = wl.random_matrix(g, 7, O, I)
    x = g.standard_normal((3, I)).astype(np.float32)
    ones = np.ones(wl.scale_count(7, O, I, 0), np.float32)
    dec = _e4m3_library(m.data)
    y64, mag = orc.matmul(7, 0, O, I, m.data, ones, x, mutation=mutation, want=("y64", "yabs"))
    want = x.astype(np.float64) @ dec.T
    if not np.all(np.abs(y64 - want) <= 1e-12 * mag):
        return False
    y2, = orc.matmul(7, 0, O, I, m.data, 2 * ones, x, mutation=mutation, want=("y64",))
    return bool(np.array_equal(y2, 2 * y64))


def _absorb_cases(g):
    """(fmt, gs, matrix, dequantized f64 matrix from raw codes / library decode)."""
    out = []
    O, I = 60, 70
    for fmt, gs in ((0, 0), (1, 0), (2, 0), (3, 0), (4, 16), (4, 6), (7, 0)):
        if fmt == 0:
            m = wl.random_matrix(g, 0, O, I)
            deq = m.data.astype(np.float64)
        elif fmt == 7:
            m = wl.random_matrix(g, 7, O, I)
            deq = _e4m3_library(m.data) * np.repeat(np.repeat(m.scales.astype(np.float64).reshape(1, 1), O, 0), I, 1)
        else:
            codes = _raw(g, fmt, O, I)
            sc = wl.log_uniform(g, 1e-3, 1e-2, wl.scale_count(fmt, O, I, gs))
            m = wl.Matrix(fmt, gs, O, I, wl.pack(fmt, codes), sc)
            deq = _deq_from_raw(fmt, gs, codes, sc)
        out.append((fmt, gs, m, deq))
    return out


def pin_absorb_vs_library(mutation=0):
    """Absorption products ([A]) on heads with a row stride larger than the rows
    per head: numpy over the matrix dequantized from raw codes (FP8: the
    library decode; its 60 x 70 shape is one scale block), forward and
    transposed, within f32 rounding."""
    g = wl.rng(20)
    o0, stride, n_rows, n_heads, S = 3, 17, 9, 3, 2
    for fmt, gs, m, deq in _absorb_cases(g):
        rows = np.array([[o0 + h * stride + j for j in range(n_rows)] for h in range(n_heads)])
        xf = g.standard_normal((S, n_heads, m.I)).astype(np.float32)
        xt = g.standard_normal((S, n_heads, n_rows)).astype(np.float32)
        want_f = np.einsum("hji,shi->shj", deq[rows], xf.astype(np.float64))
        want_t = np.einsum("hji,shj->shi", deq[rows], xt.astype(np.float64))
        mag_f = np.einsum("hji,shi->shj", np.abs(deq[rows]), np.abs(xf.astype(np.float64)))
        mag_t = np.einsum("hji,shj->shi", np.abs(deq[rows]), np.abs(xt.astype(np.float64)))
        got_f = orc.matmul_rows(fmt, gs, m.O, m.I, m.data, m.scales, o0, stride, n_rows, n_heads, xf,
                                mutation=mutation).astype(np.float64)
        got_t = orc.matmul_rows_t(fmt, gs, m.O, m.I, m.data, m.scales, o0, stride, n_rows, n_heads, xt,
                                  mutation=mutation).astype(np.float64)
        if not (np.all(np.abs(got_f - want_f) <= 2.0 ** -23 * np.abs(want_f) + 1e-12 * mag_f) and
                np.all(np.abs(got_t - want_t) <= 2.0 ** -23 * np.abs(want_t) + 1e-12 * mag_t)):
            return False
    return True


def pin_absorb_addrow_single(mutation=0):
    """One head of one row with coefficient c: the transposed product is
    c times that dequantized row (qt_addrow), element for element."""
    g = wl.rng(21)
    for fmt, gs, m, deq in _absorb_cases(g):
        for row in (0, 31, m.O - 1):
            c = np.float32(g.standard_normal())
            got = orc.matmul_rows_t(fmt, gs, m.O, m.I, m.data, m.scales, row, 0, 1, 1, np.array([[[c]]], np.float32),
                                    mutation=mutation)[0, 0].astype(np.float64)
            if not np.array_equal(got, (float(c) * deq[row]).astype(np.float32).astype(np.float64)):
                return False
    return True


def pin_absorb_adjoint(mutation=0):
    """The two absorption products are adjoint: <x_f, T(x_t)> = <F(x_f), x_t>
    for every head, within the rounding of the f32 outputs."""
    g = wl.rng(22)
    o0, stride, n_rows, n_heads = 5, 11, 11, 4
    for fmt, gs, m, _ in _absorb_cases(g):
        xf = g.standard_normal((1, n_heads, m.I)).astype(np.float32)
        xt = g.standard_normal((1, n_heads, n_rows)).astype(np.float32)
        yf = orc.matmul_rows(fmt, gs, m.O, m.I, m.data, m.scales, o0, stride, n_rows, n_heads, xf,
                             mutation=mutation).astype(np.float64)
        yt = orc.matmul_rows_t(fmt, gs, m.O, m.I, m.data, m.scales, o0, stride, n_rows, n_heads, xt,
                               mutation=mutation).astype(np.float64)
        a = np.einsum("shi,shi->sh", xf.astype(np.float64), yt)
        b = np.einsum("shj,shj->sh", yf, xt.astype(np.float64))
        scale = np.einsum("shi,shi->sh", np.abs(xf.astype(np.float64)), np.abs(yt)) + \
            np.einsum("shj,shj->sh", np.abs(yf), np.abs(xt.astype(np.float64)))
        if not np.all(np.abs(a - b) <= 1e-5 * scale):
            return False
    return True


PINS = [pin_golden_layout, pin_expert_bytes, pin_all_bytes_brute, pin_exact_integer_cases,
        pin_random_vs_library, pin_int8_unit_scale, pin_fmt4_wide_group_is_fmt2, pin_inline_order,
        pin_scale_linearity, pin_partial_last_group, pin_silu_closed_form, pin_route_vs_sorted,
        pin_moe_composition, pin_moe_invariants, pin_topk_worked_example, pin_topk_vs_sort,
        pin_fp8_block_count, pin_fp8_all_bytes, pin_fp8_block_structure, pin_fp8_unit_scale_vs_library,
        pin_absorb_vs_library, pin_absorb_addrow_single, pin_absorb_adjoint, pin_int3_golden_layout,
        pin_int3_single_codes, pin_int3_within_int4]

MUTATIONS = {
    1: "int4 nibble order swapped",
    2: "int4 read as two's complement",
    3: "fmt=4 uses a per-row scale",
    4: "fmt=4 group boundary shifted by one",
    5: "last term of the dot product dropped",
    6: "silu sign error",
    7: "routing weight dropped",
    8: "router ties go to the higher id",
    9: "router selection ignores the bias",
    10: "fmt=7 block index transposed",
    11: "fmt=7 subnormals read as normals",
    12: "absorption heads packed at n_rows instead of the row stride",
    13: "int3 codes read from the high bits of a unit first",
    14: "int3 read with offset 3 instead of 4",
}

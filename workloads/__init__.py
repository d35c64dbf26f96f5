"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and bench.py.

This module holds none of the method's arithmetic: it draws random codes,
scales, activations and routings and writes them in the documented host byte
layout (the inverse direction of decoding; it never dequantizes, multiplies or
accumulates).  Both the CPU oracle and the CUDA library consume what it
produces; neither is imported here.

Host byte layout (the library's upload input):
  fmt=0  f32 row-major [O][I]
  fmt=1  int8 two's complement, row-major [O][I]
  fmt=2  int4 offset binary (value = nibble - 8), rows of ceil(I/2) bytes,
         element 2j in the LOW nibble of byte j, element 2j+1 in the high one
  fmt=3  int2 offset binary (value = crumb - 2), rows of ceil(I/4) bytes,
         element 4j+t in bits [2t, 2t+1] of byte j
  fmt=4  as fmt=2, plus f32 scales [O][ceil(I/gs)]
  fmt=5  int3 offset binary (value = code - 4), rows of 3*ceil(I/8) bytes:
         element 8j+t is bits [3t, 3t+2] of the little-endian 24-bit word in
         bytes 3j..3j+2; f32 scales [O][ceil(I/gs)], gs a multiple of 8
  fmt=7  one FP8 E4M3 byte per element, row-major [O][I], plus f32 scales
         [ceil(O/128)][ceil(I/128)], one per 128 x 128 block
Scales are f32: [O] for fmt 1-3, [O][ceil(I/gs)] for fmt 4 and 5, per block for
fmt=7, none for fmt=0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

CODE_RANGE = {1: (-128, 127), 2: (0, 15), 3: (0, 3), 4: (0, 15), 5: (0, 7)}
OFFSET = {1: 0, 2: 8, 3: 2, 4: 8, 5: 4}
FP8_BLOCK = 128                       # fmt=7 scale block edge (rows and inputs)
FP8_NAN = (0x7F, 0xFF)                # the two E4M3 NaN bytes


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def row_bytes(fmt: int, I: int) -> int:
    return {0: 4 * I, 1: I, 2: (I + 1) // 2, 3: (I + 3) // 4, 4: (I + 1) // 2, 5: 3 * ((I + 7) // 8), 7: I}[fmt]


def n_groups(I: int, gs: int) -> int:
    return (I + gs - 1) // gs


def scale_count(fmt: int, O: int, I: int, gs: int) -> int:
    if fmt == 0:
        return 0
    if fmt in (4, 5):
        return O * n_groups(I, gs)
    if fmt == 7:
        return n_groups(O, FP8_BLOCK) * n_groups(I, FP8_BLOCK)
    return O


def tensor_bytes(fmt: int, O: int, I: int, gs: int = 0) -> int:
    """Packed codes plus f32 scales of one matrix, in host layout."""
    return O * row_bytes(fmt, I) + 4 * scale_count(fmt, O, I, gs)


def pack(fmt: int, codes: np.ndarray) -> np.ndarray:
    """Write codes [O, I] in the host byte layout.  codes are raw codes: int8
    values for fmt=1, nibbles 0..15 for fmt=2/4, crumbs 0..3 for fmt=3,
    3-bit codes 0..7 for fmt=5."""
    codes = np.asarray(codes)
    O, I = codes.shape
    if fmt == 1:
        return codes.astype(np.int8).view(np.uint8).copy()
    if fmt in (2, 4):
        c = np.zeros((O, 2 * row_bytes(fmt, I)), dtype=np.uint8)
        c[:, :I] = codes
        return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    if fmt == 3:
        c = np.zeros((O, 4 * row_bytes(fmt, I)), dtype=np.uint8)
        c[:, :I] = codes
        return (c[:, 0::4] | (c[:, 1::4] << 2) | (c[:, 2::4] << 4) | (c[:, 3::4] << 6)).astype(np.uint8)
    if fmt == 5:
        n_units = row_bytes(fmt, I) // 3
        c = np.zeros((O, 8 * n_units), dtype=np.uint32)
        c[:, :I] = codes
        word = np.zeros((O, n_units), dtype=np.uint32)
        for t in range(8):
            word |= c[:, t::8] << np.uint32(3 * t)
        out = np.empty((O, n_units, 3), dtype=np.uint8)
        for k in range(3):
            out[:, :, k] = (word >> np.uint32(8 * k)) & np.uint32(0xFF)
        return out.reshape(O, 3 * n_units)
    raise ValueError(fmt)


@dataclass
class Matrix:
    fmt: int
    gs: int
    O: int
    I: int
    data: np.ndarray            # packed bytes (uint8 [O, row_bytes]) or f32 [O, I]
    scales: np.ndarray | None   # f32

    @property
    def nbytes(self) -> int:
        return tensor_bytes(self.fmt, self.O, self.I, self.gs)


def log_uniform(g: np.random.Generator, lo: float, hi: float, n) -> np.ndarray:
    return np.exp(g.uniform(math.log(lo), math.log(hi), n)).astype(np.float32)


def random_matrix(g: np.random.Generator, fmt: int, O: int, I: int, gs: int = 0,
                  scale_lo: float = 1e-3, scale_hi: float = 1e-2) -> Matrix:
    """Uniform random codes over the format's whole code range and log-uniform
    f32 scales (the single-GEMV recipe); fmt=0 draws N(0, 0.02) weights."""
    if fmt == 0:
        return Matrix(0, 0, O, I, g.normal(0.0, 0.02, (O, I)).astype(np.float32), None)
    if fmt == 7:
        # uniform over the 254 non-NaN bytes: every finite E4M3 value, subnormals included
        v = g.integers(0, 254, (O, I))
        data = (v + (v >= 0x7F)).astype(np.uint8)   # 0..0x7E, 0x80..0xFE
        return Matrix(7, 0, O, I, data, log_uniform(g, scale_lo, scale_hi, scale_count(7, O, I, 0)))
    if fmt in (2, 4):
        # two independent uniform nibbles per byte
        data = np.frombuffer(g.bytes(O * row_bytes(fmt, I)), dtype=np.uint8).reshape(O, -1).copy()
        if I % 2:
            data[:, -1] &= 0x0F
    else:
        lo, hi = CODE_RANGE[fmt]
        data = pack(fmt, g.integers(lo, hi + 1, (O, I)))
    sc = log_uniform(g, scale_lo, scale_hi, scale_count(fmt, O, I, gs))
    return Matrix(fmt, gs, O, I, data, sc)


def quantize(fmt: int, W: np.ndarray, gs: int = 0) -> Matrix:
    """Symmetric absmax quantiser for the format sweep's N(0, 0.02) weights:
    scale = absmax / qmax per row (per group for fmt 4 and 5), qmax = 127 / 7 / 1 / 3,
    code = clip(round(w / scale)) + offset.  Input generation only."""
    W = np.asarray(W, dtype=np.float32)
    O, I = W.shape
    if fmt == 0:
        return Matrix(0, 0, O, I, W.copy(), None)
    qmax = {1: 127, 2: 7, 3: 1, 4: 7, 5: 3}[fmt]
    lo = {1: -127, 2: -8, 3: -2, 4: -8, 5: -4}[fmt]
    if fmt in (4, 5):
        ng = n_groups(I, gs)
        pad = np.zeros((O, ng * gs), dtype=np.float32)
        pad[:, :I] = W
        amax = np.abs(pad.reshape(O, ng, gs)).max(axis=2)
        sc = np.where(amax > 0, amax / qmax, 1.0).astype(np.float32)
        q = np.clip(np.rint(pad.reshape(O, ng, gs) / sc[:, :, None]), lo, qmax).reshape(O, -1)[:, :I]
        scales = sc.reshape(-1)
    else:
        amax = np.abs(W).max(axis=1)
        sc = np.where(amax > 0, amax / qmax, 1.0).astype(np.float32)
        q = np.clip(np.rint(W / sc[:, None]), lo, qmax)
        scales = sc
    codes = q.astype(np.int64) + OFFSET[fmt]
    return Matrix(fmt, gs, O, I, pack(fmt, codes), scales.astype(np.float32))


def activations(g: np.random.Generator, S: int, I: int, bf16_exact: bool = False) -> np.ndarray:
    x = g.standard_normal((S, I)).astype(np.float32)
    if bf16_exact:
        # round to the nearest bf16 value (ties to even), kept in f32
        u = x.view(np.uint32)
        u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
        x = u.astype(np.uint32).view(np.float32)
    return x


def routing_topk_softmax(g: np.random.Generator, S: int, n_experts: int, K: int):
    """Decode routing: logits N(0,1), the top-K ids (ties to the lower id) and
    the softmax of their logits (computed in double, stored as f32)."""
    logits = g.standard_normal((S, n_experts))
    ids = np.argsort(-logits, axis=1, kind="stable")[:, :K].astype(np.int32)
    top = np.take_along_axis(logits, ids.astype(np.int64), axis=1)
    e = np.exp(top - top.max(axis=1, keepdims=True))
    w = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


def routing_zipf(g: np.random.Generator, S: int, n_experts: int, K: int, s: float = 1.1):
    """Prefill routing: per row K distinct experts by successive sampling
    without replacement from Zipf(s) popularity over ranks; a seeded
    permutation maps rank -> expert id; weights = softmax of N(0,1) logits."""
    ranks = np.arange(1, n_experts + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    perm = g.permutation(n_experts)
    ids = np.empty((S, K), dtype=np.int32)
    for r in range(S):
        ids[r] = perm[g.choice(n_experts, size=K, replace=False, p=p)]
    logits = g.standard_normal((S, K))
    e = np.exp(logits - logits.max(axis=1, keepdims=True))
    w = (e / e.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# ---------------------------------------------------------------- workloads
# The five workloads of the headline benchmark.  Seeds are 1234 + index.

GEMV_SINGLE = dict(name="gemv_fmt4_single", fmt=4, S=1, I=2048, O=1536, gs=64, seed=1234)
GEMV_SWEEP = dict(name="gemv_format_sweep", I=6144, O=2048, S=(1, 2, 4),
                  variants=((0, 0), (1, 0), (2, 0), (3, 0), (4, 64), (4, 128)), seed=1235)
MOE_DECODE = dict(name="moe_decode_block", H=6144, F=2048, E=256, K=8, S=1, fmt=4, gs=64, seed=1236)
MOE_PREFILL = dict(name="moe_prefill_block", H=6144, F=2048, E=256, K=8, S=544, fmt=4, gs=128,
                   zipf=1.1, seed=1237)
STREAMING = dict(name="weight_streaming", O=2048, I=6144, pool_gb=40.0, per_layer=8, layers=75,
                 variants=((2, 0), (4, 64)), seed=1238)


def expert(g: np.random.Generator, H: int, F: int, fmt: int, gs: int):
    """(gate [F,H], up [F,H], down [H,F]) with uniform codes and log-uniform scales."""
    return (random_matrix(g, fmt, F, H, gs), random_matrix(g, fmt, F, H, gs),
            random_matrix(g, fmt, H, F, gs))


def expert_bytes(H: int, F: int, fmt: int, gs: int) -> int:
    return 2 * tensor_bytes(fmt, F, H, gs) + tensor_bytes(fmt, H, F, gs)

"""The seeded input generators produce what the input recipe states (no GPU):
shapes, code ranges, distinct Zipf routing, normalised routing weights,
bf16-exact activations, finite FP8 bytes and the packed layouts' sizes."""
import numpy as np

import workloads as wl


def test_seeded_generators_repeat():
    a = wl.random_matrix(wl.rng(5), 4, 33, 70, 16)
    b = wl.random_matrix(wl.rng(5), 4, 33, 70, 16)
    assert np.array_equal(a.data, b.data) and np.array_equal(a.scales, b.scales)


def test_matrix_shapes_and_scale_counts():
    g = wl.rng(6)
    for fmt, gs, O, I in ((0, 0, 7, 9), (1, 0, 7, 9), (2, 0, 7, 9), (3, 0, 7, 9), (4, 4, 7, 9), (7, 0, 300, 130)):
        m = wl.random_matrix(g, fmt, O, I, gs)
        if fmt == 0:
            assert m.data.shape == (O, I) and m.data.dtype == np.float32 and m.scales is None
        else:
            assert m.data.shape == (O, wl.row_bytes(fmt, I)) and m.data.dtype == np.uint8
            assert m.scales.size == wl.scale_count(fmt, O, I, gs)
            assert np.all(m.scales >= 1e-3 * (1 - 1e-6)) and np.all(m.scales <= 1e-2 * (1 + 1e-6))
    # odd int4 rows leave the unused high nibble of the last byte zero
    m = wl.random_matrix(g, 2, 5, 9)
    assert np.all(m.data[:, -1] >> 4 == 0)


def test_fp8_bytes_are_finite_and_cover_the_format():
    m = wl.random_matrix(wl.rng(7), 7, 400, 400)
    assert not np.isin(m.data, [0x7F, 0xFF]).any()
    assert len(np.unique(m.data)) == 254


def test_quantizer_codes_in_range():
    g = wl.rng(8)
    W = g.normal(0, 0.02, (16, 300)).astype(np.float32)
    for fmt, gs, lo, hi in ((1, 0, -127, 127), (2, 0, 0, 15), (3, 0, 0, 3), (4, 64, 0, 15)):
        m = wl.quantize(fmt, W, gs)
        assert m.scales.size == wl.scale_count(fmt, 16, 300, gs) and np.all(m.scales > 0)
        if fmt == 1:
            codes = m.data.view(np.int8).astype(np.int64)
        elif fmt in (2, 4):
            codes = np.stack([m.data & 0xF, m.data >> 4], axis=2).reshape(16, -1)[:, :300]
        else:
            codes = np.stack([(m.data >> (2 * t)) & 3 for t in range(4)], axis=2).reshape(16, -1)[:, :300]
        assert codes.min() >= lo and codes.max() <= hi


def test_routing_generators():
    g = wl.rng(9)
    ids, w = wl.routing_topk_softmax(g, 5, 256, 8)
    assert ids.shape == (5, 8) and ids.dtype == np.int32
    assert all(len(set(r)) == 8 for r in ids.tolist())
    assert np.allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6) and np.all(np.diff(w, axis=1) <= 0)
    ids, w = wl.routing_zipf(g, 544, 256, 8)
    assert all(len(set(r)) == 8 for r in ids.tolist()) and ids.min() >= 0 and ids.max() < 256
    assert np.allclose(w.astype(np.float64).sum(axis=1), 1.0, atol=1e-6)
    counts = np.bincount(ids.ravel(), minlength=256)
    assert counts.max() > 20 * np.median(counts[counts > 0])   # a few hot experts, a long tail


def test_bf16_exact_activations():
    x = wl.activations(wl.rng(10), 3, 1000, bf16_exact=True)
    assert np.all(x.view(np.uint32) & 0xFFFF == 0)

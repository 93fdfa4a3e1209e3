"""Pins for the oracle's blockwise quantization (CPU only).

Blockwise FP8 ("GEMM Kernel 性能优化十问", Q2): activations get one scale per
row per 128 elements, weights one scale per 128x128 block.  Per block
("实现差距：GMM Kernel（V1 vs V2）", §3.3): scale = absmax / 448,
inv = 0 if scale == 0 else 1/scale, q = e4m3(x * inv).

The pins do not retype that formula: they check closed forms (a block whose
absmax is 448 has scale exactly 1; power-of-two rescaling), the quantization
error bound of e4m3, block locality (an element only touches its own block's
scale and codes), the scale against numpy's IEEE fp32 division, and hand-
derived points (tests/golden/quant_reciprocal_points.txt) at which multiplying
by the fp32-rounded reciprocal and dividing by the scale give different codes.
"""
import os

import numpy as np
import pytest

import oracle
from fp8_blockwise_quantized_gb300.workloads import bf16_bits_to_f32, f32_to_bf16_bits


def _rand_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * np.float32(scale))


def test_lhs_shapes_and_scale_definition():
    x = _rand_bf16((37, 384), 1)
    xq, xs = oracle.quantize_lhs(x)
    assert xq.shape == (37, 384) and xs.shape == (37, 3)
    xf = bf16_bits_to_f32(x).reshape(37, 3, 128)
    amax = np.abs(xf).max(axis=2)
    # numpy float32 division is IEEE binary32 division
    assert np.array_equal(xs, (amax / np.float32(448.0)).astype(np.float32))


def test_lhs_absmax_element_maps_to_448():
    x = _rand_bf16((64, 256), 2)
    xq, xs = oracle.quantize_lhs(x)
    xf = bf16_bits_to_f32(x).reshape(64, 2, 128)
    idx = np.abs(xf).argmax(axis=2)
    q = xq.reshape(64, 2, 128)
    picked = np.take_along_axis(q, idx[..., None], axis=2)[..., 0]
    assert np.all((picked & 0x7F) == 0x7E)


def test_lhs_block_with_absmax_448_has_unit_scale():
    # every value of the block is e4m3-representable and the block max is 448
    codes = np.arange(0, 0x7F, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    rng = np.random.default_rng(3)
    row = rng.choice(vals, 128)
    row[17] = 448.0
    row *= rng.choice([-1.0, 1.0], 128)
    x = f32_to_bf16_bits(row.astype(np.float32)[None, :])
    assert np.array_equal(bf16_bits_to_f32(x)[0].astype(np.float64), row)
    xq, xs = oracle.quantize_lhs(x)
    assert xs[0, 0] == 1.0
    assert np.array_equal(oracle.e4m3_decode(xq[0]), row)


def test_lhs_zero_block():
    x = np.zeros((3, 256), np.uint16)
    x[1, 128:] = f32_to_bf16_bits(np.full(128, 0.5, np.float32))
    x[2, :128] = 0x8000  # -0.0
    xq, xs = oracle.quantize_lhs(x)
    assert xs[0, 0] == 0 and xs[0, 1] == 0 and xs[1, 0] == 0 and xs[2, 0] == 0
    assert np.all(xq[0] == 0) and np.all(xq[1, :128] == 0)
    assert np.all(xq[2, :128] == 0x80)  # sign of zero kept
    assert xs[1, 1] == np.float32(0.5) / np.float32(448.0)
    assert np.all(xq[1, 128:] == 0x7E)


def test_lhs_power_of_two_rescale_is_exact():
    x = _rand_bf16((16, 256), 4)
    xq, xs = oracle.quantize_lhs(x)
    for j in (-20, -3, 1, 9):
        x2 = f32_to_bf16_bits(bf16_bits_to_f32(x) * np.float32(2.0 ** j))
        xq2, xs2 = oracle.quantize_lhs(x2)
        assert np.array_equal(xq2, xq)
        assert np.array_equal(xs2, xs * np.float32(2.0 ** j))


def test_lhs_error_bound():
    x = _rand_bf16((128, 512), 5, scale=3.0)
    xq, xs = oracle.quantize_lhs(x)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    deq = oracle.e4m3_decode(xq) * np.repeat(xs.astype(np.float64), 128, axis=1)
    s = np.repeat(xs.astype(np.float64), 128, axis=1)
    # e4m3 rounding: half an ulp = 2^-4 relative for normals, 2^-10 absolute
    # (in units of the scale) for subnormals; plus fp32 rounding of 1/scale.
    bound = np.abs(xf) * (2.0 ** -4 + 2.0 ** -22) + s * 2.0 ** -10
    assert np.all(np.abs(deq - xf) <= bound)


def test_lhs_block_locality():
    x = _rand_bf16((8, 384), 6)
    xq, xs = oracle.quantize_lhs(x)
    x2 = x.copy()
    x2[5, 200] = f32_to_bf16_bits(np.array([1000.0], np.float32))[0]
    xq2, xs2 = oracle.quantize_lhs(x2)
    changed_s = np.argwhere(xs2 != xs)
    assert changed_s.tolist() == [[5, 1]]
    diff = np.argwhere(xq2 != xq)
    assert np.all(diff[:, 0] == 5) and np.all((diff[:, 1] >= 128) & (diff[:, 1] < 256))


def test_rhs_block_locality_and_scale():
    rng = np.random.default_rng(7)
    G, K, N = 2, 256, 384
    w = f32_to_bf16_bits((rng.standard_normal((G, K, N)) * 0.05).astype(np.float32))
    wq, ws = oracle.quantize_rhs(w)
    assert wq.shape == (G, K, N) and ws.shape == (G, 2, 3)
    wf = bf16_bits_to_f32(w).reshape(G, 2, 128, 3, 128)
    amax = np.abs(wf).max(axis=(2, 4))
    assert np.array_equal(ws, (amax / np.float32(448.0)).astype(np.float32))
    # one big element at (g=1, k=130, n=5) only moves block (1, 1, 0)
    w2 = w.copy()
    w2[1, 130, 5] = f32_to_bf16_bits(np.array([7.0], np.float32))[0]
    wq2, ws2 = oracle.quantize_rhs(w2)
    assert np.argwhere(ws2 != ws).tolist() == [[1, 1, 0]]
    d = np.argwhere(wq2 != wq)
    assert np.all(d[:, 0] == 1) and np.all((d[:, 1] >= 128) & (d[:, 1] < 256))
    assert np.all(d[:, 2] < 128)
    assert wq2[1, 130, 5] == 0x7E


def test_rhs_matches_lhs_on_a_single_block_row():
    # a 128x128 block quantized as RHS equals the LHS rule applied to the
    # block flattened into one 1x16384 group: both are absmax/448 of the block.
    rng = np.random.default_rng(8)
    w = f32_to_bf16_bits(rng.standard_normal((1, 128, 128)).astype(np.float32))
    wq, ws = oracle.quantize_rhs(w)
    xf = bf16_bits_to_f32(w).ravel()
    s = np.float32(np.abs(xf).max()) / np.float32(448.0)
    assert ws[0, 0, 0] == s


@pytest.mark.parametrize("bad", [(4, 100), (4, 0)])
def test_lhs_rejects_bad_k(bad):
    with pytest.raises(Exception):
        oracle.quantize_lhs(np.zeros(bad, np.uint16))


# ---------------------------------------------------------------------------
# multiply by the rounded reciprocal, not divide ("实现差距：GMM Kernel（V1 vs
# V2）", §3.3 takes 1/scale once and multiplies every element by it).  The
# points in tests/golden/quant_reciprocal_points.txt were derived by hand so
# that the two readings give different codes; the oracle must give the
# multiply reading's code, and each point must really separate the readings.
# ---------------------------------------------------------------------------

RECIP_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "quant_reciprocal_points.txt")


def _recip_points():
    pts = []
    for line in open(RECIP_GOLDEN):
        line = line.split("#", 1)[0].strip()
        if not line:
            continue
        a, x, mul_code, div_code = line.split()
        ev = lambda e: float(eval(e, {"__builtins__": {}}))
        pts.append((ev(a), ev(x), int(mul_code, 16), int(div_code, 16)))
    return pts


def _bits(v):
    b = f32_to_bf16_bits(np.array([v], np.float32))[0]
    assert float(bf16_bits_to_f32(np.array([b], np.uint16))[0]) == v, f"{v} is not a bf16 value"
    return b


def test_reciprocal_points_lhs():
    pts = _recip_points()
    assert len(pts) >= 12 and all(m != d for _, _, m, d in pts)
    x = np.zeros((len(pts), 256), np.uint16)
    for i, (a, v, _, _) in enumerate(pts):
        # the absmax and the probed element in block 1 of row i, at positions
        # that move with i; block 0 holds the same pair mirrored
        x[i, 128 + (i * 7) % 128] = _bits(a)
        x[i, 128 + (i * 7 + 61) % 128] = _bits(v)
        x[i, (i * 11 + 3) % 128] = _bits(-a)
        x[i, (i * 11 + 90) % 128] = _bits(v)
    xq, xs = oracle.quantize_lhs(x)
    for i, (a, v, mul, div) in enumerate(pts):
        assert xs[i, 1] == np.float32(a) / np.float32(448.0) and xs[i, 0] == xs[i, 1]
        assert xq[i, 128 + (i * 7 + 61) % 128] == mul, (a, v, hex(xq[i, 128 + (i * 7 + 61) % 128]), hex(mul))
        assert xq[i, (i * 11 + 90) % 128] == mul
        assert xq[i, 128 + (i * 7) % 128] == 0x7E and xq[i, (i * 11 + 3) % 128] == 0xFE
        assert xq[i, 128 + (i * 7 + 61) % 128] != div


def test_reciprocal_points_rhs():
    pts = _recip_points()
    G = len(pts)
    w = np.zeros((G, 128, 256), np.uint16)
    for g, (a, v, _, _) in enumerate(pts):
        w[g, (g * 5) % 128, 128 + (g * 3) % 128] = _bits(a)
        w[g, (g * 5 + 40) % 128, 128 + (g * 3 + 77) % 128] = _bits(v)
    wq, ws = oracle.quantize_rhs(w)
    for g, (a, v, mul, div) in enumerate(pts):
        assert ws[g, 0, 1] == np.float32(a) / np.float32(448.0) and ws[g, 0, 0] == 0.0
        got = wq[g, (g * 5 + 40) % 128, 128 + (g * 3 + 77) % 128]
        assert got == mul and got != div, (a, v, hex(got))
        assert wq[g, (g * 5) % 128, 128 + (g * 3) % 128] == 0x7E

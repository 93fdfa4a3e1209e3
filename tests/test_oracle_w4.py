"""Pins for the oracle's 4-bit weight path (CPU only): the FP4 E2M1 codec, the
128x128 weight quantization with scale = absmax / 6, and the forward with e2m1
weight codes ("实现差距：GMM Kernel（V1 vs V2）", §3.4: int4 / float4_e2m1fn
weights, the blockwise fp32-scale arithmetic otherwise unchanged).

The codec is pinned against hand-derived points of the format definition
(tests/golden/e2m1_points.txt), against the e4m3 codec (pinned independently
against torch's float8 cast: every e2m1 value is an e4m3 value), and against
its invariants.  The quantizer is pinned by closed forms, the e2m1 error bound,
block locality, numpy's fp32 division for the scale, and hand-derived points
where multiplying by the rounded reciprocal and dividing give different codes.
The forward is pinned by a closed form (all scales 1: the exact product of the
decoded values), by numpy's fp64 matmul on a single group, and against the
e4m3 forward fed the same weight values as e4m3 codes.
"""
import os

import numpy as np
import pytest

import oracle
from fp8_blockwise_quantized_gb300.workloads import bf16_bits_to_f32, f32_to_bf16_bits

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1_MAGS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _lines(name):
    for line in open(os.path.join(GOLDEN, name)):
        line = line.split("#", 1)[0].strip()
        if line:
            yield line.split()


def _ev(e):
    return float(eval(e, {"__builtins__": {}}))


def test_decode_table_from_the_definition():
    pts = [(int(c, 16), float(v)) for kind, c, v in _lines("e2m1_points.txt") if kind == "d"]
    assert len(pts) == 16
    got = oracle.e2m1_decode(np.array([c for c, _ in pts], np.uint8))
    for (c, v), g in zip(pts, got):
        assert g == v and np.signbit(g) == np.signbit(v), (hex(c), g, v)


def test_encode_golden_points():
    pts = [(float(v), int(c, 16)) for kind, v, c in _lines("e2m1_points.txt") if kind == "e"]
    assert len(pts) >= 20
    got = oracle.e2m1_encode(np.array([v for v, _ in pts], np.float32))
    for (v, c), g in zip(pts, got):
        assert g == c, f"encode({v}) = {g:#x}, want {c:#x}"


def test_codec_invariants():
    codes = np.arange(16, dtype=np.uint8)
    vals = oracle.e2m1_decode(codes)
    # every code round-trips, the sign is bit 3, magnitudes increase with the code
    assert np.array_equal(oracle.e2m1_encode(vals.astype(np.float32)), codes)
    assert np.array_equal(vals[8:], -vals[:8])
    assert np.all(np.diff(vals[:8]) > 0)
    # every e2m1 value is exactly an e4m3 value (the e4m3 codec is pinned
    # against torch's float8_e4m3fn cast)
    assert np.array_equal(oracle.e4m3_decode(oracle.e4m3_encode(vals.astype(np.float32))), vals)


def test_encode_is_nearest_on_a_dense_grid():
    # brute force on a dense grid: the chosen value is never farther than any
    # other code's value, and exact ties pick the even code
    v = np.linspace(-7.0, 7.0, 20001).astype(np.float32)
    c = oracle.e2m1_encode(v)
    got = oracle.e2m1_decode(c)
    allv = np.array(E2M1_MAGS + [-m for m in E2M1_MAGS])
    dist = np.abs(v.astype(np.float64)[:, None] - allv[None, :]).min(axis=1)
    clipped = np.clip(v.astype(np.float64), -6.0, 6.0)
    assert np.all(np.abs(clipped - got) <= dist + 1e-12)
    tie = np.isclose(np.abs(clipped - got), dist) & (np.sum(np.isclose(
        np.abs(v.astype(np.float64)[:, None] - allv[None, :]), dist[:, None]), axis=1) > 1)
    assert np.all((c[tie] & 1) == 0)


def _w(G, K, N, seed, scale=0.05):
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits((rng.standard_normal((G, K, N)) * scale).astype(np.float32))


def test_scale_is_absmax_over_6():
    w = _w(2, 256, 384, 1)
    wq, ws = oracle.quantize_rhs_e2m1(w)
    assert wq.shape == (2, 256, 384) and ws.shape == (2, 2, 3) and wq.max() <= 15
    amax = np.abs(bf16_bits_to_f32(w).reshape(2, 2, 128, 3, 128)).max(axis=(2, 4))
    assert np.array_equal(ws, (amax / np.float32(6.0)).astype(np.float32))


def test_block_with_absmax_6_has_unit_scale():
    rng = np.random.default_rng(2)
    vals = np.array(E2M1_MAGS)
    blk = rng.choice(vals, (128, 128)) * rng.choice([-1.0, 1.0], (128, 128))
    blk[5, 9] = 6.0
    w = f32_to_bf16_bits(blk.astype(np.float32))[None]
    wq, ws = oracle.quantize_rhs_e2m1(w)
    assert ws[0, 0, 0] == 1.0
    assert np.array_equal(oracle.e2m1_decode(wq[0]), blk)


def test_zero_block_and_power_of_two_rescale():
    w = _w(1, 128, 256, 3)
    w[0, :, 128:] = 0
    wq, ws = oracle.quantize_rhs_e2m1(w)
    assert ws[0, 0, 1] == 0 and np.all(wq[0, :, 128:] == 0)
    for j in (-9, 2, 11):
        w2 = f32_to_bf16_bits(bf16_bits_to_f32(w) * np.float32(2.0 ** j))
        wq2, ws2 = oracle.quantize_rhs_e2m1(w2)
        assert np.array_equal(wq2, wq) and np.array_equal(ws2, ws * np.float32(2.0 ** j))


def test_error_bound():
    w = _w(2, 256, 256, 4, scale=1.0)
    wq, ws = oracle.quantize_rhs_e2m1(w)
    s = np.repeat(np.repeat(ws.astype(np.float64), 128, axis=1), 128, axis=2)
    deq = oracle.e2m1_decode(wq) * s
    wf = bf16_bits_to_f32(w).astype(np.float64)
    # half the e2m1 spacing: 1/4 relative for normals (one mantissa bit),
    # 1/4 of the scale for the subnormal 0.5; plus the fp32 reciprocal
    bound = np.abs(wf) * (2.0 ** -2 + 2.0 ** -22) + s * 2.0 ** -2
    assert np.all(np.abs(deq - wf) <= bound)


def test_block_locality():
    w = _w(2, 256, 256, 5)
    wq, ws = oracle.quantize_rhs_e2m1(w)
    w2 = w.copy()
    w2[1, 200, 7] = f32_to_bf16_bits(np.array([9.0], np.float32))[0]
    wq2, ws2 = oracle.quantize_rhs_e2m1(w2)
    assert np.argwhere(ws2 != ws).tolist() == [[1, 1, 0]]
    d = np.argwhere(wq2 != wq)
    assert np.all(d[:, 0] == 1) and np.all(d[:, 1] >= 128) and np.all(d[:, 2] < 128)
    assert wq2[1, 200, 7] == 0x7


def test_reciprocal_points():
    pts = [(_ev(a), _ev(x), int(m, 16), int(d, 16)) for a, x, m, d in _lines("quant_reciprocal_points_e2m1.txt")]
    assert len(pts) >= 8 and all(m != d for _, _, m, d in pts)
    G = len(pts)
    w = np.zeros((G, 128, 128), np.uint16)
    for g, (a, v, _, _) in enumerate(pts):
        for val in (a, v):
            b = f32_to_bf16_bits(np.array([val], np.float32))[0]
            assert float(bf16_bits_to_f32(np.array([b], np.uint16))[0]) == val
        w[g, (g * 3) % 128, (g * 7) % 128] = f32_to_bf16_bits(np.array([a], np.float32))[0]
        w[g, (g * 3 + 50) % 128, (g * 7 + 33) % 128] = f32_to_bf16_bits(np.array([v], np.float32))[0]
    wq, ws = oracle.quantize_rhs_e2m1(w)
    for g, (a, v, mul, div) in enumerate(pts):
        assert ws[g, 0, 0] == np.float32(a) / np.float32(6.0)
        got = wq[g, (g * 3 + 50) % 128, (g * 7 + 33) % 128]
        assert got == mul and got != div, (a, v, hex(got))
        assert wq[g, (g * 3) % 128, (g * 7) % 128] == 0x7


def _xq_unit_scale(M, K, rng):
    """Activations whose every 1x128 block has absmax 448 and e4m3 values:
    the quantized codes decode to the values themselves, scale 1."""
    vals = oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    x = rng.choice(vals[vals <= 32.0], (M, K)) * rng.choice([-1.0, 1.0], (M, K))
    x[:, ::128] = 448.0
    return f32_to_bf16_bits(x.astype(np.float32)), x


def test_forward_closed_form_with_unit_scales():
    rng = np.random.default_rng(6)
    sizes = np.array([3, 0, 5, 2], np.int32)
    M, K, N = 12, 256, 128
    xb, xv = _xq_unit_scale(M, K, rng)
    wv = rng.choice(E2M1_MAGS, (4, K, N)) * rng.choice([-1.0, 1.0], (4, K, N))
    wv[:, ::128, 0] = 6.0
    xq, xs = oracle.quantize_lhs(xb)
    wq, ws = oracle.quantize_rhs_e2m1(f32_to_bf16_bits(wv.astype(np.float32)))
    assert np.all(xs == 1.0) and np.all(ws == 1.0)
    out = oracle.gmm_fp8_w4(xq, xs, wq, ws, sizes)
    off = np.concatenate([[0], np.cumsum(sizes)])
    for g in range(4):
        exact = xv[off[g]:off[g + 1]] @ wv[g]
        assert np.array_equal(out[off[g]:off[g + 1]], exact)
    assert np.all(out[off[-1]:] == 0)


def test_forward_single_group_equals_dequantized_matmul():
    rng = np.random.default_rng(7)
    M, K, N = 9, 384, 256
    x = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = _w(1, K, N, 8, scale=0.1)
    xq, xs = oracle.quantize_lhs(x)
    wq, ws = oracle.quantize_rhs_e2m1(w)
    out = oracle.gmm_fp8_w4(xq, xs, wq, ws, np.array([M], np.int32))
    xd = oracle.e4m3_decode(xq) * np.repeat(xs.astype(np.float64), 128, axis=1)
    wd = oracle.e2m1_decode(wq[0]) * np.repeat(np.repeat(ws[0].astype(np.float64), 128, axis=0), 128, axis=1)
    ref = np.matmul(xd, wd)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


@pytest.mark.parametrize("fuse", [False, True])
def test_forward_equals_the_e4m3_forward_on_the_same_values(fuse):
    # e2m1 values are e4m3 values: re-encoding the weight codes as e4m3 (with
    # the same scales) must give the e4m3 forward's result bit for bit
    rng = np.random.default_rng(9)
    sizes = np.array([70, 0, 130, 1], np.int32)
    M, K, N = 211, 256, 128
    x = f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    w = _w(4, K, 2 * N if fuse else N, 10, scale=0.08)
    xq, xs = oracle.quantize_lhs(x)
    wq4, ws = oracle.quantize_rhs_e2m1(w)
    wq8 = oracle.e4m3_encode(oracle.e2m1_decode(wq4).astype(np.float32))
    a = oracle.gmm_fp8_w4(xq, xs, wq4, ws, sizes, fuse=fuse)
    b = oracle.gmm_fp8(xq, xs, wq8, ws, sizes, fuse=fuse)
    assert np.array_equal(a, b)

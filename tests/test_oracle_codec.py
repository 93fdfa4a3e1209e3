"""Pins for the oracle's e4m3 and bf16 codecs (CPU only).

The oracle's codec is written from the E4M3 format definition.  It is pinned
here against (a) hand-derived points of that definition (tests/golden), (b) an
independent library implementation (torch's float8_e4m3fn cast) over every
bf16 bit pattern, and (c) structural invariants of the format.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_points.txt")


def _golden_points():
    pts = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            expr, code = line.split()
            pts.append((float(eval(expr, {"__builtins__": {}})), int(code, 16)))
    return pts


def test_golden_points():
    pts = _golden_points()
    assert len(pts) >= 20
    vals = np.array([p[0] for p in pts], np.float32)
    codes = oracle.e4m3_encode(vals)
    for (v, c), got in zip(pts, codes):
        assert got == c, f"encode({v}) = {got:#x}, want {c:#x}"


def test_decode_definition_landmarks():
    d = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert d[0x38] == 1.0 and d[0x7E] == 448.0 and d[0x08] == 2.0 ** -6
    assert d[0x01] == 2.0 ** -9 and d[0x07] == 7 * 2.0 ** -9
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.count_nonzero(np.isnan(d)) == 2
    # sign symmetry
    assert np.array_equal(d[:0x7F], -d[0x80:0xFF]) or np.all((d[:0x7F] == -d[0x80:0xFF]))
    # finite non-negative codes are strictly increasing in value
    assert np.all(np.diff(d[:0x7F]) > 0)
    # 8 values per binade in the normal range
    assert d[0x10] / d[0x08] == 2.0 and d[0x18] / d[0x10] == 2.0


def test_roundtrip_all_finite_codes():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)


def test_matches_torch_cast_on_every_bf16_pattern():
    # Library cross-check: torch's float8_e4m3fn cast rounds to nearest even;
    # it returns NaN at |v| >= 464 where the method saturates (never reached by
    # the quantizer, whose |x * inv| <= 448 up to fp32 rounding).
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    finite = np.isfinite(vals) & (np.abs(vals) < 464.0)
    v = vals[finite]
    mine = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(mine, ref)


def test_matches_torch_cast_on_fp32_midpoints():
    # exact midpoints between adjacent e4m3 values exercise ties-to-even
    d = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((d[:-1] + d[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, 0), np.nextafter(mids, 1000)])
    near = np.concatenate([near, -near])
    ref = torch.from_numpy(near.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(near), ref)


def test_saturation_and_nan():
    v = np.array([448.0, 449.0, 463.99, 464.0, 1e30, np.inf, -np.inf, np.nan], np.float32)
    c = oracle.e4m3_encode(v)
    assert list(c[:6]) == [0x7E] * 6
    assert c[6] == 0xFE
    assert c[7] == 0x7F


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000),
        # exact bf16 midpoints in fp64 (ties) and their neighbours
        ((np.arange(1, 2000) * 2 + 1) * 2.0 ** -8),
    ])
    ref = torch.from_numpy(v).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(oracle.round_to_bf16(v), ref.view(np.uint16))


def test_bf16_widen_is_exact():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    ok = ~np.isnan(ref)
    assert np.array_equal(f[ok], ref[ok])


def test_silu_matches_library():
    xs = np.linspace(-30, 30, 1201)
    mine = np.array([oracle.silu(v) for v in xs])
    ref = torch.nn.functional.silu(torch.from_numpy(xs)).numpy()
    np.testing.assert_allclose(mine, ref, rtol=1e-14, atol=1e-300)
    assert oracle.silu(0.0) == 0.0

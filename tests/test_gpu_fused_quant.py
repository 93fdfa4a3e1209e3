"""GPU parity of the fused SwiGLU + FP8-cast epilogue (gmm_fp8_fwd_swiglu_quant).

The fused kernel must write exactly what quantizing its own bf16 h with
gmm_quantize_lhs gives (checked bit for bit, GPU against GPU), and its h must
match the oracle as the plain fused forward does.  Against the oracle, the
1x128 blocks whose bf16 h equals the oracle's bit for bit must also have the
oracle's codes and scale bit for bit; the remaining blocks (an accumulation-
order ulp in h) must dequantize to within the e4m3 rounding bound of the
oracle's h.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import normal_bf16
from tests.gpu_util import FP8_ATOL, FP8_RTOL, Guarded, assert_close, bf16_to_np64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

CASES = [
    ([512], 512, 256, 256),
    ([0, 300, 0, 212], 600, 256, 384),
    ([1, 127, 128, 129, 0, 2], 400, 384, 256),
    ([5, 0, 0, 9], 14, 256, 128),
]


def _check_against_oracle(x, w, s, h, hq, hs):
    """h against the oracle; hq/hs bit for bit on the 1x128 blocks whose h
    equals the oracle's, within the e4m3 bound elsewhere; zero tail rows."""
    M, N = h.shape
    S = int(s.sum())
    assert torch.all(hq[S:] == 0) and torch.all(hs[:, S:] == 0)
    oxq, oxs = oracle.quantize_lhs(x)
    owq, ows = oracle.quantize_rhs(w)
    h_ref = oracle.gmm_fp8(oxq, oxs, owq, ows, s, fuse=True)
    got_h = bf16_to_np64(h)
    assert_close(got_h, h_ref, FP8_ATOL, FP8_RTOL, "fused h")
    h_bits = oracle.round_to_bf16(h_ref)
    ohq, ohs = oracle.quantize_lhs(h_bits)
    gh_bits = h.view(torch.int16).cpu().numpy().view(np.uint16)
    ghq = hq.cpu().numpy()
    ghs = hs.cpu().numpy().T
    same = (gh_bits.reshape(M, N // 128, 128) == h_bits.reshape(M, N // 128, 128)).all(axis=2)
    assert same.mean() > 0.5
    blk_q = ghq.reshape(M, N // 128, 128)
    assert np.array_equal(blk_q[same], ohq.reshape(M, N // 128, 128)[same])
    assert np.array_equal(ghs[same].view(np.uint32), ohs[same].view(np.uint32))
    deq = oracle.e4m3_decode(ghq) * np.repeat(ghs.astype(np.float64), 128, axis=1)
    hb = oracle.bf16_to_f64(h_bits)
    bound = np.abs(hb) * 2.0 ** -4 + np.repeat(ghs.astype(np.float64), 128, axis=1) * 2.0 ** -9 + \
        FP8_ATOL + FP8_RTOL * np.abs(hb)
    assert np.all(np.abs(deq - hb) <= bound)


def _guarded_outputs(M, N):
    return (Guarded((M, N), torch.bfloat16), Guarded((M, N), torch.uint8),
            Guarded((N // 128, M), torch.float32))


@pytest.mark.parametrize("sizes,M,K,N", CASES)
def test_fused_quant(sizes, M, K, N):
    rng = np.random.default_rng(M + 5 * K + N)
    s = np.array(sizes, np.int32)
    G = len(sizes)
    x = normal_bf16((M, K), 1.0, rng, outlier_p=0.01)
    w = normal_bf16((G, K, 2 * N), 1.0 / np.sqrt(K), rng)
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    wq, ws = gmm.quantize_rhs(to_dev_bf16(w))
    sd = to_dev(s)
    g = _guarded_outputs(M, N)
    h, hq, hs = gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, sd, out=tuple(b.t for b in g))
    _, hq2, hs2 = gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, sd, with_h=False)
    rq, rs = gmm.quantize_lhs(h)
    torch.cuda.synchronize()
    for b, what in zip(g, ("h", "hq", "hs")):
        b.check(f"fused quant {what}")
    # GPU consistency: fused == quantize(h), and without h the same bits
    assert torch.equal(hq, rq) and torch.equal(hs.view(torch.int32), rs.view(torch.int32))
    assert torch.equal(hq, hq2) and torch.equal(hs.view(torch.int32), hs2.view(torch.int32))
    _check_against_oracle(x, w, s, h, hq, hs)


@pytest.mark.parametrize("ctas,order,cg", [(5, 1, 1), (9, 2, 1), (4, 1, 2), (8, 2, 2), (0, 1, 0)])
def test_fused_quant_many_units_per_cta(ctas, order, cg):
    """A mid-size problem with few persistent CTAs (or CTA pairs, cg = 2), so
    that every CTA runs many work units back to back: the staging area, its
    free/staged barriers, the TMEM buffers and the scale ring change phase
    across units, against the oracle (ctas = 0: the default launch)."""
    rng = np.random.default_rng(4000 + ctas)
    G, M, K, N = 9, 4000, 512, 512
    s = rng.multinomial(M - 37, np.full(G, 1.0 / G)).astype(np.int32)
    s[0] += s[3]  # group 3 empty, group 7 a single row
    s[3] = 0
    s[7] = 1
    M_rows = int(s.sum()) + 37  # 37 tail rows past the last group
    x = normal_bf16((M_rows, K), 1.0, rng, outlier_p=0.01)
    w = normal_bf16((G, K, 2 * N), 1.0 / np.sqrt(K), rng)
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    wq, ws = gmm.quantize_rhs(to_dev_bf16(w))
    g = _guarded_outputs(M_rows, N)
    cfg = (256, ctas, order, cg) if ctas else None
    h, hq, hs = gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, to_dev(s), out=tuple(b.t for b in g), config=cfg)
    torch.cuda.synchronize()
    for b, what in zip(g, ("h", "hq", "hs")):
        b.check(f"fused quant {what}")
    rows_per_tile = 256 if cg == 2 else 128
    units = sum((int(n) + rows_per_tile - 1) // rows_per_tile for n in s) * (N // 128)
    assert ctas == 0 or units * (2 if cg == 2 else 1) >= 12 * ctas
    _check_against_oracle(x, w, s, h, hq, hs)

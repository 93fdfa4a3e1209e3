"""Pins for the oracle's grouped GEMMs and group metadata (CPU only).

A grouped GEMM is one independent GEMM per expert over that expert's
contiguous rows ("MoE 优化的探索", §3.7.2); rows past sum(group_sizes) are
zero ("实现差距：GMM Kernel（V1 vs V2）", §3.6).  The FP8 forward rescales each
128-wide K partial by the LHS row scale and the RHS block scale
("GEMM Kernel 性能优化十问", Q1/Q3; §3.3 of the V1/V2 page); tgmm is
dW[g] = X_g^T dY_g (Q4), in bf16 (Q5).

Pins: brute force on tiny inputs, closed forms with unit scales (exact integer
results), library matmuls of dequantized operands (torch fp64), torch's silu,
and invariants (permutation, exact power-of-two scaling, empty groups, zero
tail, the sum identity of tgmm).
"""
import numpy as np
import pytest
import torch

import oracle
from fp8_blockwise_quantized_gb300.workloads import (bf16_bits_to_f32, f32_to_bf16_bits,
                                                     subproblem_sizes)


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16(a):
    return f32_to_bf16_bits(np.asarray(a, np.float32))


def _dequant_x(xq, xs):
    return oracle.e4m3_decode(xq) * np.repeat(xs.astype(np.float64), 128, axis=1)


def _dequant_w(wq, ws):
    s = np.repeat(np.repeat(ws.astype(np.float64), 128, axis=1), 128, axis=2)
    return oracle.e4m3_decode(wq) * s


def _torch_group_mm(a, b, sizes, fuse=False):
    """Library reference: torch fp64 matmul per group on dense operands."""
    M = a.shape[0]
    Nw = b.shape[2]
    N = Nw // 2 if fuse else Nw
    out = np.zeros((M, N))
    off = np.concatenate([[0], np.cumsum(sizes)])
    for g in range(len(sizes)):
        r0, r1 = off[g], off[g + 1]
        if r1 == r0:
            continue
        y = torch.from_numpy(a[r0:r1]) @ torch.from_numpy(b[g])
        if fuse:
            y = torch.nn.functional.silu(y[:, :N]) * y[:, N:]
        out[r0:r1] = y.numpy()
    return out


# ----------------------------------------------------------------------------
# metadata
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("sizes,M,bm", [
    ([3, 0, 5], 8, 2), ([0, 0, 0], 4, 128), ([129, 127, 128, 1, 0, 256], 700, 128),
    ([1], 1, 128), ([300], 300, 64),
])
def test_tiles_brute_force(sizes, M, bm):
    off, tiles = oracle.group_tiles(np.array(sizes, np.int32), M, bm)
    # brute force: walk the rows one by one
    want = []
    row = 0
    for g, n in enumerate(sizes):
        for i in range(0, n, bm):
            want.append((g, row + i, row + min(i + bm, n)))
        row += n
    assert [tuple(t) for t in tiles.tolist()] == want
    assert off.tolist() == [0] + list(np.cumsum(sizes))
    assert len(tiles) <= (M + bm - 1) // bm + len(sizes)


def test_metadata_errors():
    with pytest.raises(oracle.OracleError) as e:
        oracle.group_offsets(np.array([3, -1, 2], np.int32), 10)
    assert e.value.status == oracle.ERR_NEGATIVE_GROUP
    with pytest.raises(oracle.OracleError) as e:
        oracle.group_offsets(np.array([3, 8], np.int32), 10)
    assert e.value.status == oracle.ERR_GROUPS_EXCEED_M


# ----------------------------------------------------------------------------
# FP8 GMM
# ----------------------------------------------------------------------------

def test_fp8_tiny_hand_computed():
    # X row m is the constant c_m, W[g] the constant d_g: every block's absmax
    # is |c| (|d|), so every code is 448 and the result is
    # K * 448^2 * fl32(c/448) * fl32(d/448) for each output element.
    sizes = np.array([2, 0, 3], np.int32)
    M, K, N = 5, 128, 128
    c = np.array([1.0, -0.5, 3.0, 0.25, 2.0], np.float32)
    d = np.array([0.125, 7.0, -1.5], np.float32)
    x = _bf16(np.repeat(c[:, None], K, axis=1))
    w = _bf16(np.broadcast_to(d[:, None, None], (3, K, N)))
    xq, xs = oracle.quantize_lhs(x)
    wq, ws = oracle.quantize_rhs(w)
    y = oracle.gmm_fp8(xq, xs, wq, ws, sizes)
    grp = [0, 0, 2, 2, 2]
    for m in range(M):
        sx = np.float64(np.float32(abs(c[m])) / np.float32(448))
        sw = np.float64(np.float32(abs(d[grp[m]])) / np.float32(448))
        want = K * 448.0 * 448.0 * sx * sw * np.sign(c[m]) * np.sign(d[grp[m]])
        assert np.all(y[m] == want)


def test_fp8_unit_scales_exact_integer_result():
    # scales 1 and integer-valued codes: the grouped product is an exact
    # integer matmul (numpy int64, a library routine).
    rng = _rng(11)
    all_vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    ints = np.array([c for c, v in enumerate(all_vals) if v == np.floor(v) and v <= 16], np.uint8)
    assert len(ints) == 17  # every integer 0..16 is an e4m3 value
    sizes = np.array([7, 0, 5, 4], np.int32)
    M, K, N, G = 20, 256, 256, 4
    xq = rng.choice(ints, (M, K)) | (rng.integers(0, 2, (M, K)) * 0x80).astype(np.uint8)
    wq = rng.choice(ints, (G, K, N)) | (rng.integers(0, 2, (G, K, N)) * 0x80).astype(np.uint8)
    xs = np.ones((M, K // 128), np.float32)
    ws = np.ones((G, K // 128, N // 128), np.float32)
    y = oracle.gmm_fp8(xq, xs, wq, ws, sizes)
    xi = oracle.e4m3_decode(xq).astype(np.int64)
    wi = oracle.e4m3_decode(wq).astype(np.int64)
    off = np.concatenate([[0], np.cumsum(sizes)])
    want = np.zeros((M, N), np.int64)
    for g in range(G):
        want[off[g]:off[g + 1]] = xi[off[g]:off[g + 1]] @ wi[g]
    assert np.array_equal(y, want.astype(np.float64))
    assert np.all(y[off[-1]:] == 0)


@pytest.mark.parametrize("fuse", [False, True])
def test_fp8_equals_library_matmul_of_dequantized(fuse):
    # The blockwise definition equals the plain product of the dequantized
    # operands (fp64): this pins every scale index (row, k-block, n-block, g).
    rng = _rng(12 + fuse)
    G, K, N = 3, 384, 256
    sizes = np.array([70, 0, 51], np.int32)
    M = 130  # two tail rows past sum(sizes)
    Nw = 2 * N if fuse else N
    x = _bf16(rng.standard_normal((M, K)) * np.exp(rng.standard_normal((M, 1))))
    w = _bf16(rng.standard_normal((G, K, Nw)) * np.exp(rng.standard_normal((G, 1, Nw))) / 20)
    xq, xs = oracle.quantize_lhs(x)
    wq, ws = oracle.quantize_rhs(w)
    y = oracle.gmm_fp8(xq, xs, wq, ws, sizes, fuse=fuse)
    ref = _torch_group_mm(_dequant_x(xq, xs), _dequant_w(wq, ws), sizes, fuse=fuse)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.all(y[121:] == 0)


def test_fp8_single_group_is_plain_gemm():
    rng = _rng(14)
    M, K, N = 64, 256, 128
    x = _bf16(rng.standard_normal((M, K)))
    w = _bf16(rng.standard_normal((1, K, N)) / 16)
    xq, xs = oracle.quantize_lhs(x)
    wq, ws = oracle.quantize_rhs(w)
    y = oracle.gmm_fp8(xq, xs, wq, ws, np.array([M], np.int32))
    ref = (torch.from_numpy(_dequant_x(xq, xs)) @ torch.from_numpy(_dequant_w(wq, ws)[0])).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_fp8_group_permutation_and_scaling():
    rng = _rng(15)
    G, K, N = 3, 256, 128
    sizes = np.array([5, 9, 3], np.int32)
    M = 17
    x = _bf16(rng.standard_normal((M, K)))
    w = _bf16(rng.standard_normal((G, K, N)) / 16)
    xq, xs = oracle.quantize_lhs(x)
    wq, ws = oracle.quantize_rhs(w)
    y = oracle.gmm_fp8(xq, xs, wq, ws, sizes)
    # permute groups (2, 0, 1) with their row blocks
    perm = [2, 0, 1]
    off = np.concatenate([[0], np.cumsum(sizes)])
    rows = np.concatenate([np.arange(off[g], off[g + 1]) for g in perm])
    y2 = oracle.gmm_fp8(xq[rows], xs[rows], wq[perm], ws[perm], sizes[perm])
    assert np.array_equal(y2, y[rows])
    # W[1] * 2: the scales double exactly, the codes stay, the rows double
    w2 = w.copy()
    w2[1] = _bf16(bf16_bits_to_f32(w[1]) * 2)
    wq2, ws2 = oracle.quantize_rhs(w2)
    assert np.array_equal(wq2, wq) and np.array_equal(ws2[1], ws[1] * 2)
    y3 = oracle.gmm_fp8(xq, xs, wq2, ws2, sizes)
    assert np.array_equal(y3[5:14], 2 * y[5:14])
    assert np.array_equal(y3[:5], y[:5]) and np.array_equal(y3[14:], y[14:])


def test_fp8_empty_groups_and_zero_tail():
    rng = _rng(16)
    G, K, N = 4, 128, 128
    M = 40
    x = _bf16(rng.standard_normal((M, K)))
    w = _bf16(rng.standard_normal((G, K, N)))
    xq, xs = oracle.quantize_lhs(x)
    wq, ws = oracle.quantize_rhs(w)
    y0 = oracle.gmm_fp8(xq, xs, wq, ws, np.zeros(G, np.int32))
    assert np.all(y0 == 0)
    sizes = np.array([0, 10, 0, 20], np.int32)
    y = oracle.gmm_fp8(xq, xs, wq, ws, sizes)
    assert np.all(y[30:] == 0) and np.any(y[:30] != 0)
    # the empty groups' weights do not matter
    wq_b = wq.copy()
    wq_b[0] = 0x38
    wq_b[2] = 0x38
    assert np.array_equal(oracle.gmm_fp8(xq, xs, wq_b, ws, sizes), y)


def test_fp8_sampled_rows_subproblem():
    # The tests compare full-size outputs on sampled rows by running the GMM on
    # the sampled rows alone with per-group counts: pin that this equals the
    # same rows of the full problem.
    rng = _rng(17)
    G, K, N = 3, 256, 128
    sizes = np.array([9, 0, 12], np.int32)
    M = 21
    x = _bf16(rng.standard_normal((M, K)))
    w = _bf16(rng.standard_normal((G, K, N)))
    xq, xs = oracle.quantize_lhs(x)
    wq, ws = oracle.quantize_rhs(w)
    y = oracle.gmm_fp8(xq, xs, wq, ws, sizes)
    rows = np.array([0, 4, 8, 9, 15, 20])
    sub = subproblem_sizes(sizes, rows)
    assert sub.tolist() == [3, 0, 3]
    ys = oracle.gmm_fp8(xq[rows], xs[rows], wq, ws, sub)
    assert np.array_equal(ys, y[rows])


def test_fp8_rejects_bad_groups():
    xq = np.zeros((4, 128), np.uint8)
    xs = np.zeros((4, 1), np.float32)
    wq = np.zeros((2, 128, 128), np.uint8)
    ws = np.zeros((2, 1, 1), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.gmm_fp8(xq, xs, wq, ws, np.array([3, 2], np.int32))
    with pytest.raises(oracle.OracleError):
        oracle.gmm_fp8(xq, xs, wq, ws, np.array([-1, 2], np.int32))


# ----------------------------------------------------------------------------
# bf16 GMM and tgmm
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("fuse", [False, True])
def test_bf16_gmm_equals_library(fuse):
    rng = _rng(20 + fuse)
    G, K, N = 3, 192, 128
    sizes = np.array([33, 0, 60], np.int32)
    M = 100
    Nw = 2 * N if fuse else N
    x = _bf16(rng.standard_normal((M, K)))
    w = _bf16(rng.standard_normal((G, K, Nw)) / 8)
    y = oracle.gmm_bf16(x, w, sizes, fuse=fuse)
    ref = _torch_group_mm(bf16_bits_to_f32(x).astype(np.float64),
                          bf16_bits_to_f32(w).astype(np.float64), sizes, fuse=fuse)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.all(y[93:] == 0)


def test_bf16_gmm_unquantized_matches_fp8_when_exact():
    # values representable in e4m3 with unit block scales: the FP8 GMM and the
    # bf16 GMM compute the same exact numbers.
    rng = _rng(22)
    G, K, N = 2, 256, 128
    sizes = np.array([6, 6], np.int32)
    codes = np.arange(0, 0x70, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    xv = rng.choice(vals, (12, K))
    wv = rng.choice(vals, (G, K, N)) / 448.0 * 448.0
    xv[:, ::128] = 448.0
    wv[:, ::128, ::128] = 448.0
    wv[:, 0, :] = 448.0
    xq, xs = oracle.quantize_lhs(_bf16(xv))
    wq, ws = oracle.quantize_rhs(_bf16(wv))
    assert np.all(xs == 1) and np.all(ws == 1)
    a = oracle.gmm_fp8(xq, xs, wq, ws, sizes)
    b = oracle.gmm_bf16(_bf16(xv), _bf16(wv), sizes)
    assert np.array_equal(a, b)


def test_tgmm_equals_library_and_sum_identity():
    rng = _rng(23)
    G, K, N = 4, 128, 256
    sizes = np.array([10, 0, 25, 7], np.int32)
    M = 45
    x = _bf16(rng.standard_normal((M, K)))
    dy = _bf16(rng.standard_normal((M, N)))
    dw = oracle.tgmm_bf16(x, dy, sizes)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    df = bf16_bits_to_f32(dy).astype(np.float64)
    off = np.concatenate([[0], np.cumsum(sizes)])
    for g in range(G):
        ref = (torch.from_numpy(xf[off[g]:off[g + 1]]).T @ torch.from_numpy(df[off[g]:off[g + 1]])).numpy()
        np.testing.assert_allclose(dw[g], ref, rtol=1e-12, atol=1e-12)
    assert np.all(dw[1] == 0)
    S = off[-1]
    total = (torch.from_numpy(xf[:S]).T @ torch.from_numpy(df[:S])).numpy()
    np.testing.assert_allclose(dw.sum(axis=0), total, rtol=1e-10, atol=1e-10)
    # rows past S do not contribute
    x2 = x.copy()
    x2[S:] = _bf16(np.full((M - S, K), 99.0))
    assert np.array_equal(oracle.tgmm_bf16(x2, dy, sizes), dw)


def test_tgmm_tiny_brute_force():
    # G=2, M=3, K=N=1 style hand computation embedded in 128-wide arrays
    x = np.zeros((3, 128), np.float32)
    dy = np.zeros((3, 128), np.float32)
    x[:, 0] = [1.0, 2.0, 3.0]
    dy[:, 5] = [4.0, -1.0, 0.5]
    dw = oracle.tgmm_bf16(_bf16(x), _bf16(dy), np.array([2, 1], np.int32))
    assert dw[0, 0, 5] == 1 * 4 + 2 * -1
    assert dw[1, 0, 5] == 3 * 0.5
    assert np.count_nonzero(dw) == 2


def test_dgrad_equals_library_and_transposed_forward():
    # dX_g = dY_g W[g]^T: a library matmul per group, and the bf16 forward GMM
    # of dY with the transposed weights (a different oracle routine)
    rng = _rng(24)
    G, K, N = 3, 256, 384
    sizes = np.array([20, 0, 33], np.int32)
    M = 60
    dy = _bf16(rng.standard_normal((M, N)))
    w = _bf16(rng.standard_normal((G, K, N)) / 8)
    dx = oracle.dgrad_bf16(dy, w, sizes)
    wt = np.ascontiguousarray(w.transpose(0, 2, 1))
    ref = _torch_group_mm(bf16_bits_to_f32(dy).astype(np.float64), bf16_bits_to_f32(wt).astype(np.float64), sizes)
    np.testing.assert_allclose(dx, ref, rtol=1e-12, atol=1e-12)
    assert np.array_equal(dx, oracle.gmm_bf16(dy, wt, sizes))
    assert np.all(dx[53:] == 0)

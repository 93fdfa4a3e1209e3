"""GPU parity of the 4-bit weight path ("实现差距：GMM Kernel（V1 vs V2）", §3.4:
float4_e2m1fn weights with the blockwise fp32-scale arithmetic kept) against
the oracle: the E2M1 weight quantization bit for bit (codes and scale bits),
the FP8 x FP4 forward element by element on ragged, empty and tail-row cases,
plain and fused, the fused FP8 cast of h, the CTA-pair kernel's bits, the
development shape in full and the production shape on sampled rows.

Tolerance: the FP8 bound of the other forward tests (atol 1e-3, rtol 1e-2
against the oracle on the same codes): only the accumulation order differs."""
import numpy as np
import pytest
import torch

import oracle
import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import make_case, normal_bf16, sample_rows, subproblem_sizes
from tests.gpu_util import FP8_ATOL, FP8_RTOL, Guarded, assert_close, bf16_to_np64, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

EDGE = [
    ([512], 512, 256, 256),
    ([0, 300, 0, 212], 512, 256, 256),
    ([1, 127, 128, 129, 0, 2], 400, 384, 384),
    ([130, 0, 150], 300, 128, 128),
    ([5, 0, 0, 9], 14, 256, 512),
    ([0, 0, 0], 64, 256, 256),
]


def _unpack(wq4):
    """[G, N, K/2] packed codes -> [G, K, N] one code per byte (the oracle's layout)."""
    b = wq4.cpu().numpy()
    codes = np.stack([b & 0xF, b >> 4], axis=-1).reshape(b.shape[0], b.shape[1], -1)
    return np.ascontiguousarray(codes.transpose(0, 2, 1))


def test_quantize_w4_bit_exact():
    rng = np.random.default_rng(44)
    G, K, N = 3, 384, 256
    w = normal_bf16((G, K, N), 0.05, rng, outlier_p=0.01)
    w[1, 128:256, 128:] = 0  # an all-zero block
    wq4, ws = gmm.quantize_rhs_w4(to_dev_bf16(w))
    torch.cuda.synchronize()
    owq, ows = oracle.quantize_rhs_e2m1(w)
    assert np.array_equal(_unpack(wq4), owq)
    assert np.array_equal(ws.cpu().numpy().view(np.uint32), ows.view(np.uint32))


def _run(s, x, w, fuse, cfg=None):
    M, K = x.shape
    G, _, Nw = w.shape
    N = Nw // 2 if fuse else Nw
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    wq4, ws = gmm.quantize_rhs_w4(to_dev_bf16(w))
    out = Guarded((M, N), torch.bfloat16)
    work = gmm.Workspace(G, M)
    gmm.fp8_w4_fwd(xq, xs, wq4, ws, to_dev(s), fuse=fuse, out=out.t, workspace=work, config=cfg)
    torch.cuda.synchronize()
    assert work.status() == 0
    out.check("fp8 x fp4 forward output")
    return out.t


def _oracle(s, x, w, fuse):
    oxq, oxs = oracle.quantize_lhs(x)
    owq, ows = oracle.quantize_rhs_e2m1(w)
    return oracle.gmm_fp8_w4(oxq, oxs, owq, ows, s, fuse=fuse)


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("sizes,M,K,N", EDGE)
def test_w4_edges(sizes, M, K, N, fuse):
    rng = np.random.default_rng(M + K + N + 7)
    s = np.array(sizes, np.int32)
    x = normal_bf16((M, K), 1.0, rng, outlier_p=0.01)
    w = normal_bf16((len(sizes), K, 2 * N if fuse else N), 1.0 / np.sqrt(K), rng)
    got = _run(s, x, w, fuse)
    ref = _oracle(s, x, w, fuse)
    assert_close(bf16_to_np64(got), ref, FP8_ATOL, FP8_RTOL, "fp8 x fp4 forward")
    assert torch.all(got[int(s.sum()):] == 0)
    if fuse or N % 256 == 0:
        # the CTA-pair kernel gives the same bits
        got2 = _run(s, x, w, fuse, cfg=(0, 0, 0, 2))
        assert torch.equal(got.view(torch.int16), got2.view(torch.int16))


def test_w4_fused_cast():
    rng = np.random.default_rng(91)
    sizes, M, K, N = [0, 300, 1, 211], 600, 256, 384
    s = np.array(sizes, np.int32)
    x = normal_bf16((M, K), 1.0, rng, outlier_p=0.01)
    w = normal_bf16((len(sizes), K, 2 * N), 1.0 / np.sqrt(K), rng)
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    wq4, ws = gmm.quantize_rhs_w4(to_dev_bf16(w))
    h, hq, hs = gmm.fp8_w4_fwd_swiglu_quant(xq, xs, wq4, ws, to_dev(s))
    rq, rs = gmm.quantize_lhs(h)
    h2 = gmm.fp8_w4_fwd(xq, xs, wq4, ws, to_dev(s), fuse=True)
    torch.cuda.synchronize()
    # the cast equals quantizing the kernel's own h, and h equals the plain fused forward's
    assert torch.equal(hq, rq) and torch.equal(hs.view(torch.int32), rs.view(torch.int32))
    assert torch.equal(h.view(torch.int16), h2.view(torch.int16))
    assert_close(bf16_to_np64(h), _oracle(s, x, w, True), FP8_ATOL, FP8_RTOL, "fp8 x fp4 fused h")


def test_w4_dev_shape_full():
    c = make_case("wi_dev_fp8")
    got = bf16_to_np64(_run(c.group_sizes, c.x, c.w, False))
    ref = _oracle(c.group_sizes, c.x, c.w, False)
    assert_close(got, ref, FP8_ATOL, FP8_RTOL, "fp8 x fp4 dev shape")
    exact = oracle.gmm_bf16(c.x, c.w, c.group_sizes)
    s_k = oracle.sqnr_db(exact, got)
    s_o = oracle.sqnr_db(exact, oracle.bf16_to_f64(oracle.round_to_bf16(ref)))
    print(f"fp8 x fp4 dev shape SQNR: kernel {s_k:.2f} dB, oracle {s_o:.2f} dB")
    assert s_k >= s_o - 0.1


def test_w4_prod_fused_cast_sampled():
    """The production wi shape (G=256, M=65536, K=2048, W 2x512 columns) with
    4-bit weights and the fused FP8 cast, on sampled rows of a dozen experts."""
    c = make_case("prod_fp8", with_second_layer=False)
    rng = np.random.default_rng(77)
    xq, xs = gmm.quantize_lhs(to_dev_bf16(c.x))
    wq4, ws = gmm.quantize_rhs_w4(to_dev_bf16(c.w))
    h, hq, hs = gmm.fp8_w4_fwd_swiglu_quant(xq, xs, wq4, ws, to_dev(c.group_sizes))
    torch.cuda.synchronize()
    live = np.flatnonzero(c.group_sizes)
    groups = sorted({int(live[np.argmax(c.group_sizes[live])]), int(live[np.argmin(c.group_sizes[live])])} |
                    {int(g) for g in rng.choice(live, 10, replace=False)})
    rows = sample_rows(c.group_sizes, 5, rng)
    off = np.concatenate([[0], np.cumsum(c.group_sizes.astype(np.int64))])
    g_of = np.searchsorted(off, rows, side="right") - 1
    rows = rows[np.isin(g_of, groups)]
    sub = subproblem_sizes(c.group_sizes, rows)[groups]
    oxq, oxs = oracle.quantize_lhs(c.x[rows])
    owq, ows = oracle.quantize_rhs_e2m1(c.w[groups])
    h_ref = oracle.gmm_fp8_w4(oxq, oxs, owq, ows, sub, fuse=True)
    rsel = torch.from_numpy(rows).cuda()
    assert_close(bf16_to_np64(h[rsel]), h_ref, FP8_ATOL, FP8_RTOL, "fp8 x fp4 production wi (sampled rows)")
    rq, rs = gmm.quantize_lhs(h)
    torch.cuda.synchronize()
    assert torch.equal(hq, rq) and torch.equal(hs.view(torch.int32), rs.view(torch.int32))

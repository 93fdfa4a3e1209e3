"""GPU parity of the grouped forward GEMMs (FP8 blockwise and bf16) against the
oracle, element by element, on ragged, empty and tail-row cases that span
several tiles, and on the two full development shapes."""
import numpy as np
import pytest
import torch

import oracle
import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import make_case, normal_bf16
from tests.gpu_util import (BF16_ATOL, BF16_RTOL, FP8_ATOL, FP8_RTOL, Guarded, assert_close, bf16_to_np64,
                            poison_bf16, to_dev, to_dev_bf16)

pytestmark = pytest.mark.gpu

# (sizes, M, K, N): empty first / middle / last groups, sizes 1, 127, 128, 129,
# sum < M (tail rows), M not a multiple of 128, one group, 128- and 256-wide
# column tiles, a single 128-wide K block.
EDGE = [
    ([512], 512, 256, 256),
    ([0, 300, 0, 212], 512, 256, 256),
    ([1, 127, 128, 129, 0, 2], 400, 384, 384),
    ([130, 0, 150], 300, 128, 128),
    ([5, 0, 0, 9], 14, 256, 512),
    ([0, 0, 0], 64, 256, 256),
    ([77, 300, 1, 255, 256, 33], 1000, 512, 640),
]


def _inputs(sizes, M, K, Nw, seed):
    rng = np.random.default_rng(seed)
    s = np.array(sizes, np.int32)
    x = normal_bf16((M, K), 1.0, rng, outlier_p=0.01)
    w = normal_bf16((len(sizes), K, Nw), 1.0 / np.sqrt(K), rng)
    return s, x, w


def _bf16_round(v):
    return oracle.bf16_to_f64(oracle.round_to_bf16(v))


def _run_fp8(s, x, w, fuse, both_kernels=False):
    M, K = x.shape
    G, _, Nw = w.shape
    N = Nw // 2 if fuse else Nw
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    wq, ws = gmm.quantize_rhs(to_dev_bf16(w))
    out = Guarded((M, N), torch.bfloat16)
    work = gmm.Workspace(G, M)
    gmm.fp8_fwd(xq, xs, wq, ws, to_dev(s), fuse=fuse, out=out.t, workspace=work)
    torch.cuda.synchronize()
    assert work.status() == 0
    out.check("fp8 fwd output")
    if both_kernels and (fuse or N % 256 == 0):
        # the CTA-pair kernel (256-row tiles) gives the default's bits
        out2 = Guarded((M, N), torch.bfloat16)
        gmm.fp8_fwd(xq, xs, wq, ws, to_dev(s), fuse=fuse, out=out2.t, workspace=work, config=(0, 0, 0, 2))
        torch.cuda.synchronize()
        assert work.status() == 0
        out2.check("fp8 fwd output, CTA pairs")
        assert torch.equal(out.t.view(torch.int16), out2.t.view(torch.int16)), "CTA pairs vs one CTA per tile"
    return bf16_to_np64(out.t)


def _oracle_fp8(s, x, w, fuse):
    oxq, oxs = oracle.quantize_lhs(x)
    owq, ows = oracle.quantize_rhs(w)
    return oracle.gmm_fp8(oxq, oxs, owq, ows, s, fuse=fuse)


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("sizes,M,K,N", EDGE)
def test_fp8_edges(sizes, M, K, N, fuse):
    if fuse and N % 128:
        pytest.skip("fused output needs N % 128 == 0")
    s, x, w = _inputs(sizes, M, K, 2 * N if fuse else N, M + K + N)
    got = _run_fp8(s, x, w, fuse, both_kernels=True)
    ref = _oracle_fp8(s, x, w, fuse)
    assert_close(got, ref, FP8_ATOL, FP8_RTOL, "fp8 fwd")
    S = int(s.sum())
    assert np.all(got[S:] == 0), "rows past sum(group_sizes) must be zero"


@pytest.mark.parametrize("scale", [40.0, 400.0])
def test_fp8_fused_extreme_gates(scale):
    """Gate values far into both tails of silu (|gate| up to ~1e3 and beyond
    the -80 clamp of the kernel's silu), with an up factor of either sign."""
    sizes, M, K, N = [200, 0, 185], 512, 256, 256
    rng = np.random.default_rng(int(scale))
    s = np.array(sizes, np.int32)
    x = normal_bf16((M, K), scale, rng)
    w = normal_bf16((len(sizes), K, 2 * N), 1.0 / np.sqrt(K), rng)
    got = _run_fp8(s, x, w, True)
    ref = _oracle_fp8(s, x, w, True)
    assert np.max(np.abs(ref)) > 100.0 and np.min(ref) < 0.0
    assert_close(got, ref, FP8_ATOL, FP8_RTOL, "fused fp8 fwd, extreme gates")


@pytest.mark.parametrize("fuse", [False, True])
@pytest.mark.parametrize("sizes,M,K,N", EDGE)
def test_bf16_edges(sizes, M, K, N, fuse):
    s, x, w = _inputs(sizes, M, K, 2 * N if fuse else N, M + K + N + 1)
    G = len(sizes)
    out = Guarded((M, N), torch.bfloat16)
    work = gmm.Workspace(G, M)
    gmm.bf16_fwd(to_dev_bf16(x), to_dev_bf16(w), to_dev(s), fuse=fuse, out=out.t, workspace=work)
    torch.cuda.synchronize()
    assert work.status() == 0
    out.check("bf16 fwd output")
    ref = oracle.gmm_bf16(x, w, s, fuse=fuse)
    assert_close(bf16_to_np64(out.t), ref, BF16_ATOL, BF16_RTOL, "bf16 fwd")


def test_fp8_tiny_config():
    c = make_case("tiny_fp8")
    assert c.group_sizes[2] == 0 and c.group_sizes.sum() == c.M
    got = _run_fp8(c.group_sizes, c.x, c.w, False)
    ref = _oracle_fp8(c.group_sizes, c.x, c.w, False)
    assert_close(got, ref, FP8_ATOL, FP8_RTOL, "tiny fp8")
    # SQNR against the unquantized fp64 product: the kernel adds no error
    # beyond the method's own (oracle SQNR minus 0.1 dB at most)
    exact = oracle.gmm_bf16(c.x, c.w, c.group_sizes)
    assert oracle.sqnr_db(exact, got) >= oracle.sqnr_db(exact, _bf16_round(ref)) - 0.1


@pytest.mark.parametrize("name", ["wi_dev_fp8", "wo_dev_fp8"])
def test_fp8_dev_shapes_full(name):
    c = make_case(name)
    got = _run_fp8(c.group_sizes, c.x, c.w, False)
    ref = _oracle_fp8(c.group_sizes, c.x, c.w, False)
    assert_close(got, ref, FP8_ATOL, FP8_RTOL, name)
    exact = oracle.gmm_bf16(c.x, c.w, c.group_sizes)
    s_kernel = oracle.sqnr_db(exact, got)
    s_oracle = oracle.sqnr_db(exact, _bf16_round(ref))
    print(f"{name}: SQNR kernel {s_kernel:.2f} dB, oracle {s_oracle:.2f} dB")
    assert s_kernel >= s_oracle - 0.1
    assert s_kernel > 30.0


def test_bf16_dev_shape_full():
    c = make_case("wi_dev_fp8")
    out = gmm.bf16_fwd(to_dev_bf16(c.x), to_dev_bf16(c.w), to_dev(c.group_sizes))
    torch.cuda.synchronize()
    ref = oracle.gmm_bf16(c.x, c.w, c.group_sizes)
    assert_close(bf16_to_np64(out), ref, BF16_ATOL, BF16_RTOL, "bf16 dev")


def test_repeated_calls_reuse_workspace():
    s, x, w = _inputs([100, 0, 200, 212], 512, 256, 256, 5)
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    wq, ws = gmm.quantize_rhs(to_dev_bf16(w))
    work = gmm.Workspace(4, 512)
    a = gmm.fp8_fwd(xq, xs, wq, ws, to_dev(s), workspace=work)
    b = gmm.fp8_fwd(xq, xs, wq, ws, to_dev(s), workspace=work)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert work.status() == 0


def test_claim_counters_shared_across_launches():
    """The FP8 forward (one CTA per tile) and tgmm both claim their units from
    the workspace's counter words and their last CTA resets them: a chain of
    launches of both kinds on one workspace, reusing its metadata (group sizes
    NULL), gives every launch the same bits as a fresh workspace, and the
    counters are zero at the end."""
    s, x, w = _inputs([700, 0, 3, 1300, 129, 0, 64], 2400, 512, 512, 11)
    G, M = len(s), 2400
    xd = to_dev_bf16(x)
    xq, xs = gmm.quantize_lhs(xd)
    wq, ws = gmm.quantize_rhs(to_dev_bf16(w))
    dy = torch.randn(M, 256, device="cuda", generator=torch.Generator(device="cuda").manual_seed(3)).to(torch.bfloat16)
    ref_y = gmm.fp8_fwd(xq, xs, wq, ws, to_dev(s), workspace=gmm.Workspace(G, M))
    ref_h = gmm.fp8_fwd(xq, xs, wq, ws, to_dev(s), workspace=gmm.Workspace(G, M), fuse=True)
    ref_dw = gmm.tgmm(xd, dy, to_dev(s), workspace=gmm.Workspace(G, M))
    work = gmm.group_metadata(to_dev(s), M)
    for _ in range(3):
        y = gmm.fp8_fwd(xq, xs, wq, ws, None, workspace=work)
        dw = gmm.tgmm(xd, dy, None, workspace=work)
        h = gmm.fp8_fwd(xq, xs, wq, ws, None, workspace=work, fuse=True)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref_y.view(torch.int16))
        assert torch.equal(h.view(torch.int16), ref_h.view(torch.int16))
        assert torch.equal(dw.view(torch.int16), ref_dw.view(torch.int16))
    assert work.status() == 0
    words = work.buf[:32].view(torch.int32).cpu()
    assert int(words[4]) == 0 and int(words[5]) == 0, "claim counters not reset"

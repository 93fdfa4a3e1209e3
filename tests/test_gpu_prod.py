"""Parity at the production shape (G=256, M=65536, K=2048, N=2x512 fused wi,
then wo K=512 N=2048, bf16 tgmm of both), in the launch configuration the
benchmark times.  The oracle cannot redo the whole layer in seconds, so it
recomputes sampled outputs: a set of experts (the largest, the smallest
non-empty one and random others), a few rows of each (always the first and
the last row of the group, where row tiles are ragged) and, for tgmm, a few
rows of dW over every column.  Each sample is itself a small grouped problem
that the oracle solves from the same inputs; nothing computed on the GPU is
fed to the oracle.  Properties that hold at any size (bit-exact quantization
of the sampled rows, zero dW for empty experts) are checked as well."""
import numpy as np
import pytest
import torch

import oracle
import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import (make_case, normal_bf16, routing_sizes, sample_rows,
                                                     subproblem_sizes)
from tests.gpu_util import (BF16_ATOL, BF16_RTOL, FP8_ATOL, FP8_RTOL, assert_close, bf16_to_np64, to_dev,
                            to_dev_bf16)

pytestmark = [pytest.mark.gpu]


@pytest.fixture(scope="module")
def prod():
    return make_case("prod_fp8")


def _pick_groups(sizes, n, rng):
    live = np.flatnonzero(sizes)
    pick = {int(live[np.argmax(sizes[live])]), int(live[np.argmin(sizes[live])])}
    rest = [g for g in live if g not in pick]
    pick.update(int(g) for g in rng.choice(rest, n - len(pick), replace=False))
    return sorted(pick)


def _restrict(sizes, groups, rows_per_group, rng):
    """Sampled rows (sorted) of the picked groups only, and the sub-problem's sizes."""
    rows = sample_rows(sizes, rows_per_group, rng)
    off = np.concatenate([[0], np.cumsum(sizes.astype(np.int64))])
    g_of = np.searchsorted(off, rows, side="right") - 1
    rows = rows[np.isin(g_of, groups)]
    sub = subproblem_sizes(sizes, rows)[groups]
    assert sub.sum() == rows.size and np.all(sub > 0)
    return rows, sub


def test_prod_forward_chain_sampled(prod):
    c = prod
    rng = np.random.default_rng(31)
    assert c.group_sizes.sum() == c.M and np.count_nonzero(c.group_sizes == 0) == 8
    G, M, K, N = c.G, c.M, c.K, c.N
    # ---- GPU: the path exactly as the benchmark runs it
    sizes_d = to_dev(c.group_sizes)
    x_d = to_dev_bf16(c.x)
    xq, xs = gmm.quantize_lhs(x_d)
    wq_wi, ws_wi = gmm.quantize_rhs(to_dev_bf16(c.w))
    wq_wo, ws_wo = gmm.quantize_rhs(to_dev_bf16(c.w2))
    work = gmm.Workspace(G, M)
    h = gmm.fp8_fwd(xq, xs, wq_wi, ws_wi, sizes_d, fuse=True, workspace=work)
    hq, hs = gmm.quantize_lhs(h)
    y = gmm.fp8_fwd(hq, hs, wq_wo, ws_wo, sizes_d, workspace=work)
    torch.cuda.synchronize()
    assert work.status() == 0

    # ---- oracle on a sample
    groups = _pick_groups(c.group_sizes, 12, rng)
    rows, sub = _restrict(c.group_sizes, groups, 6, rng)
    ox = c.x[rows]
    oxq, oxs = oracle.quantize_lhs(ox)
    assert np.array_equal(xq[torch.from_numpy(rows).cuda()].cpu().numpy(), oxq)
    assert np.array_equal(xs.t()[torch.from_numpy(rows).cuda()].cpu().numpy().view(np.uint32),
                          oxs.view(np.uint32))
    owq_wi, ows_wi = oracle.quantize_rhs(c.w[groups])
    owq_wo, ows_wo = oracle.quantize_rhs(c.w2[groups])
    gsel = torch.tensor(groups, device="cuda")
    assert np.array_equal(wq_wi[gsel].cpu().numpy().transpose(0, 2, 1), owq_wi)
    assert np.array_equal(ws_wo[gsel].cpu().numpy().view(np.uint32), ows_wo.view(np.uint32))

    h_ref = oracle.gmm_fp8(oxq, oxs, owq_wi, ows_wi, sub, fuse=True)
    rsel = torch.from_numpy(rows).cuda()
    assert_close(bf16_to_np64(h[rsel]), h_ref, FP8_ATOL, FP8_RTOL, "prod wi fused (sampled rows)")
    h_bits = oracle.round_to_bf16(h_ref)
    ohq, ohs = oracle.quantize_lhs(h_bits)
    y_ref = oracle.gmm_fp8(ohq, ohs, owq_wo, ows_wo, sub)
    assert_close(bf16_to_np64(y[rsel]), y_ref, FP8_ATOL, FP8_RTOL, "prod wo (sampled rows)")
    # SQNR of the sampled rows against the unquantized fp64 chain, kernel vs oracle
    h_exact = oracle.gmm_bf16(ox, c.w[groups], sub, fuse=True)
    s_k = oracle.sqnr_db(h_exact, bf16_to_np64(h[rsel]))
    s_o = oracle.sqnr_db(h_exact, oracle.bf16_to_f64(h_bits))
    print(f"prod wi sampled SQNR: kernel {s_k:.2f} dB, oracle {s_o:.2f} dB")
    assert s_k >= s_o - 0.1


@pytest.mark.parametrize("layer", ["wo", "wi"])
def test_prod_tgmm_sampled(layer):
    # tgmm at the production shapes of both weight gradients, on synthetic
    # activations of the same shapes (the benchmark feeds h and X)
    sizes = routing_sizes("prod_fp8")
    G, M = 256, 65536
    Kd, Nd = (512, 2048) if layer == "wo" else (2048, 1024)
    rng = np.random.default_rng(41 if layer == "wo" else 42)
    x = normal_bf16((M, Kd), 1.0, rng)
    dy = normal_bf16((M, Nd), 1.0, rng)
    dw = gmm.tgmm(to_dev_bf16(x), to_dev_bf16(dy), to_dev(sizes))
    torch.cuda.synchronize()
    dead = np.flatnonzero(sizes == 0)
    assert len(dead) == 8
    assert torch.all(dw[torch.from_numpy(dead).cuda()] == 0)
    groups = _pick_groups(sizes, 6, rng)
    ks = np.sort(rng.choice(Kd, 24, replace=False))
    ks[0], ks[-1] = 0, Kd - 1
    off = np.concatenate([[0], np.cumsum(sizes.astype(np.int64))])
    for g in groups:
        r0, r1 = off[g], off[g + 1]
        ref = oracle.tgmm_bf16(np.ascontiguousarray(x[r0:r1][:, ks]), dy[r0:r1], np.array([r1 - r0], np.int32))[0]
        got = bf16_to_np64(dw[g][torch.from_numpy(ks).cuda()])
        assert_close(got, ref, BF16_ATOL, BF16_RTOL, f"prod tgmm {layer} g={g}")

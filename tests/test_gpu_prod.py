"""Parity at the production shape (G=256, M=65536, K=2048, N=2x512 fused wi,
then wo K=512 N=2048, bf16 tgmm of both).

test_prod_bench_step_sampled runs the benchmark's step exactly: the same C
entry points with the same arguments, in the same order, on one workspace
(quantize X, one metadata pass, the fused wi writing h and its FP8 cast with
group_sizes = NULL, wo on that cast, tgmm dW_wo = h^T dY and dW_wi = X^T dH,
both with group_sizes = NULL).  The other tests check the plain fused forward
followed by a separate quantization, and tgmm at both production shapes.

The oracle cannot redo the whole layer in seconds, so it recomputes sampled
outputs: a set of experts (the largest, the smallest non-empty one and random
others), a few rows of each (always the first and the last row of the group,
where row tiles are ragged) and, for tgmm, a few rows of dW over every column.
Each sample is itself a small grouped problem that the oracle solves from the
same host inputs; nothing computed on the GPU is fed to the oracle (dW_wo,
whose input h is a GPU result, is checked against a second, standalone tgmm
launch on the GPU instead, bit for bit).  Properties that hold at any size
(bit-exact quantization of the sampled rows, zero dW for empty experts, the
tgmm work counters back at zero) are checked as well."""
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
    gh_bits = h[rsel].view(torch.int16).cpu().numpy().view(np.uint16)
    same = (gh_bits.reshape(-1, N // 128, 128) == h_bits.reshape(-1, N // 128, 128)).all(axis=2)
    _check_wo_rows(bf16_to_np64(y[rsel]), y_ref, same, oracle.bf16_to_f64(h_bits), c, groups, sub, "prod wo")
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


def _check_wo_rows(got_y, y_ref, same, hb, c, groups, sub, what):
    """wo output on sampled rows.  Rows whose FP8 cast of h equals the
    oracle's in every 1x128 block got the oracle's input: the FP8 bound holds
    as it stands.  In a row with a block whose h differs by an accumulation-
    order ulp, that block's cast differs too; each dequantized input then
    differs by at most the two e4m3 roundings (2^-4 |h| each) plus the h
    difference (within the FP8 bound), which bounds the change of y by that
    sum times |W| over the block (|W_q| <= |W| (1 + 2^-4))."""
    row_same = same.all(axis=1)
    assert row_same.mean() > 0.5
    assert_close(got_y[row_same], y_ref[row_same], FP8_ATOL, FP8_RTOL, f"{what} (sampled rows)")
    off_s = np.concatenate([[0], np.cumsum(sub.astype(np.int64))])
    g_of_row = np.searchsorted(off_s, np.arange(got_y.shape[0]), side="right") - 1
    for i in np.flatnonzero(~row_same):
        dh_max = (2.0 ** -3 * np.abs(hb[i]) + 2 * (FP8_ATOL + FP8_RTOL * np.abs(hb[i]))) * np.repeat(~same[i], 128)
        w_abs = np.abs(oracle.bf16_to_f64(c.w2[groups[g_of_row[i]]])) * (1 + 2.0 ** -4)
        bound_y = dh_max @ w_abs + FP8_ATOL + FP8_RTOL * np.abs(y_ref[i])
        assert np.all(np.abs(got_y[i] - y_ref[i]) <= bound_y), f"{what}, sampled row {i}"


def _ref_sampled_chain(c, groups, rows, sub):
    """Oracle h (fp64), its bf16 bits, the oracle's FP8 cast of h, and the
    oracle wo output for the sampled rows; plus the unquantized fp64 chain."""
    ox = c.x[rows]
    oxq, oxs = oracle.quantize_lhs(ox)
    owq_wi, ows_wi = oracle.quantize_rhs(c.w[groups])
    owq_wo, ows_wo = oracle.quantize_rhs(c.w2[groups])
    h_ref = oracle.gmm_fp8(oxq, oxs, owq_wi, ows_wi, sub, fuse=True)
    h_bits = oracle.round_to_bf16(h_ref)
    ohq, ohs = oracle.quantize_lhs(h_bits)
    y_ref = oracle.gmm_fp8(ohq, ohs, owq_wo, ows_wo, sub)
    # unquantized chain in fp64: silu(gate) * up, then wo, no rounding between
    h_exact = oracle.gmm_bf16(ox, c.w[groups], sub, fuse=True)
    off = np.concatenate([[0], np.cumsum(sub.astype(np.int64))])
    y_exact = np.empty((rows.size, c.w2.shape[2]), np.float64)
    for j in range(len(groups)):
        w2 = oracle.bf16_to_f64(c.w2[groups[j]])
        y_exact[off[j]:off[j + 1]] = h_exact[off[j]:off[j + 1]] @ w2
    return dict(oxq=oxq, oxs=oxs, h_ref=h_ref, h_bits=h_bits, ohq=ohq, ohs=ohs, y_ref=y_ref,
                h_exact=h_exact, y_exact=y_exact)


def test_prod_bench_step_sampled(prod):
    c = prod
    G, M, K, N = c.G, c.M, c.K, c.N
    rng = np.random.default_rng(57)
    dy = normal_bf16((M, K), 1.0, rng)
    dh = normal_bf16((M, 2 * N), 1.0, rng)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    chk = gmm.binding._check
    sizes = to_dev(c.group_sizes)
    x = to_dev_bf16(c.x)
    dy_d, dh_d = to_dev_bf16(dy), to_dev_bf16(dh)
    wq_wi, ws_wi = gmm.quantize_rhs(to_dev_bf16(c.w))
    wq_wo, ws_wo = gmm.quantize_rhs(to_dev_bf16(c.w2))
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    xs = torch.empty((K // 128, M), dtype=torch.float32, device=dev)
    h = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    hq = torch.empty((M, N), dtype=torch.uint8, device=dev)
    hs = torch.empty((N // 128, M), dtype=torch.float32, device=dev)
    y = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    dw_wo = torch.empty((G, N, K), dtype=torch.bfloat16, device=dev)
    dw_wi = torch.empty((G, K, 2 * N), dtype=torch.bfloat16, device=dev)
    work = gmm.Workspace(G, M, dev)
    # ---- the benchmark's step, call for call
    chk(gmm.gmm_quantize_lhs(x, M, K, xq, xs, stream), "quantize X")
    chk(gmm.gmm_group_metadata(sizes, G, M, work.buf, work.nbytes, stream), "metadata")
    chk(gmm.gmm_fp8_fwd_swiglu_quant(xq, xs, wq_wi, ws_wi, None, G, M, K, N, h, hq, hs, work.buf, work.nbytes,
                                     stream), "wi")
    chk(gmm.gmm_fp8_fwd(hq, hs, wq_wo, ws_wo, None, G, M, N, K, 0, y, work.buf, work.nbytes, stream), "wo")
    chk(gmm.tgmm_bf16(h, dy_d, None, G, M, N, K, dw_wo, work.buf, work.nbytes, stream), "tgmm wo")
    chk(gmm.tgmm_bf16(x, dh_d, None, G, M, K, 2 * N, dw_wi, work.buf, work.nbytes, stream), "tgmm wi")
    torch.cuda.synchronize()
    assert work.status() == 0
    assert work.buf[16:24].view(torch.int32).tolist() == [0, 0]  # tgmm work counters back at zero
    # dW_wo against a standalone tgmm launch with its own metadata (same kernel, same inputs: same bits)
    dw_wo2 = gmm.tgmm(h, dy_d, sizes)
    torch.cuda.synchronize()
    assert torch.equal(dw_wo.view(torch.int16), dw_wo2.view(torch.int16))
    dead = torch.from_numpy(np.flatnonzero(c.group_sizes == 0)).cuda()
    assert torch.all(dw_wo[dead] == 0) and torch.all(dw_wi[dead] == 0)

    # ---- oracle on a sample
    groups = _pick_groups(c.group_sizes, 12, rng)
    rows, sub = _restrict(c.group_sizes, groups, 6, rng)
    r = _ref_sampled_chain(c, groups, rows, sub)
    rsel = torch.from_numpy(rows).cuda()
    assert np.array_equal(xq[rsel].cpu().numpy(), r["oxq"])
    assert np.array_equal(xs.t()[rsel].cpu().numpy().view(np.uint32), r["oxs"].view(np.uint32))
    got_h = bf16_to_np64(h[rsel])
    assert_close(got_h, r["h_ref"], FP8_ATOL, FP8_RTOL, "bench step: wi h (sampled rows)")
    # the FP8 cast of h: bit for bit on the blocks whose h equals the oracle's
    gh_bits = h[rsel].view(torch.int16).cpu().numpy().view(np.uint16)
    ghq = hq[rsel].cpu().numpy()
    ghs = hs.t()[rsel].cpu().numpy()
    nb = N // 128
    same = (gh_bits.reshape(-1, nb, 128) == r["h_bits"].reshape(-1, nb, 128)).all(axis=2)
    assert same.mean() > 0.5
    assert np.array_equal(ghq.reshape(-1, nb, 128)[same], r["ohq"].reshape(-1, nb, 128)[same])
    assert np.array_equal(ghs[same].view(np.uint32), r["ohs"][same].view(np.uint32))
    deq = oracle.e4m3_decode(ghq) * np.repeat(ghs.astype(np.float64), 128, axis=1)
    hb = oracle.bf16_to_f64(r["h_bits"])
    bound = np.abs(hb) * 2.0 ** -4 + np.repeat(ghs.astype(np.float64), 128, axis=1) * 2.0 ** -9 + \
        FP8_ATOL + FP8_RTOL * np.abs(hb)
    assert np.all(np.abs(deq - hb) <= bound)
    got_y = bf16_to_np64(y[rsel])
    _check_wo_rows(got_y, r["y_ref"], same, hb, c, groups, sub, "bench step: wo y")
    # SQNR against the unquantized fp64 chain: the kernels add no error beyond the method's
    s_wi_k = oracle.sqnr_db(r["h_exact"], got_h)
    s_wi_o = oracle.sqnr_db(r["h_exact"], hb)
    s_wo_k = oracle.sqnr_db(r["y_exact"], got_y)
    s_wo_o = oracle.sqnr_db(r["y_exact"], oracle.bf16_to_f64(oracle.round_to_bf16(r["y_ref"])))
    print(f"bench step SQNR: wi kernel {s_wi_k:.2f} / oracle {s_wi_o:.2f} dB; "
          f"wo chain kernel {s_wo_k:.2f} / oracle {s_wo_o:.2f} dB")
    assert s_wi_k >= s_wi_o - 0.1
    assert s_wo_k >= s_wo_o - 0.1
    # tgmm dW_wi = X^T dH (host inputs) on sampled experts and k rows.  This
    # X carries the 1% x50 outliers, so a few dW elements are sums of
    # thousands of terms that cancel to almost nothing (terms summing to 7000
    # in absolute value, result 0.1).  Any fp32 accumulator is off there by a
    # few fp32 units of the terms' absolute sum; the bound adds 2^-18 (64
    # units) of that sum to the tgmm tolerance.
    ks = np.sort(rng.choice(K, 24, replace=False))
    ks[0], ks[-1] = 0, K - 1
    off = np.concatenate([[0], np.cumsum(c.group_sizes.astype(np.int64))])
    ksel = torch.from_numpy(ks).cuda()
    for g in groups[:6]:
        r0, r1 = off[g], off[g + 1]
        xg = np.ascontiguousarray(c.x[r0:r1][:, ks])
        ref = oracle.tgmm_bf16(xg, dh[r0:r1], np.array([r1 - r0], np.int32))[0]
        l1 = np.abs(oracle.bf16_to_f64(xg)).T @ np.abs(oracle.bf16_to_f64(dh[r0:r1]))
        got = bf16_to_np64(dw_wi[g][ksel])
        bound = BF16_ATOL + BF16_RTOL * np.abs(ref) + 2.0 ** -18 * l1
        bad = np.abs(got - ref) > bound
        assert not np.any(bad), f"bench step: dW_wi g={g}: {int(bad.sum())} elements out of tolerance"

"""Randomized GPU sweep over shapes and routings (property tests beside the
oracle parity tests).

Each case draws G, M, K, N, a routing (uniform, one huge group, Zipf-like, mostly
empty with tiny groups, or sizes at and around multiples of 16/64/128/256, the
total at most M) and bf16 data, then checks:
- the FP8 forward, plain or with the fused silu(gate)*up, is bit-identical across
  tile configurations (default, CTA pairs, bn 128, a five-CTA grid in column-block
  order) and within the FP8 bound of an fp32 matmul of the dequantized operands
  (the same codes and scales, so only the accumulation order and the final bf16
  rounding differ); rows past the groups are zero;
- the fused cast equals quantizing the kernel's own h, and h equals the fused
  forward's output;
- 4-bit weights: CTA pairs bit-identical to one CTA per tile, and the result within
  the FP8 bound of the fp32 matmul of the dequantized E2M1 weights;
- tgmm is deterministic run to run and within its bound of an fp32 X_g^T dY_g.
"""
import math

import numpy as np
import pytest
import torch

import fp8_blockwise_quantized_gb300 as gmm

pytestmark = pytest.mark.gpu

E2M1 = [0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6]


def _sizes(rng, G, M):
    kind = rng.integers(0, 5)
    if kind == 0:
        s = rng.multinomial(int(M * rng.uniform(0.5, 1.0)), np.ones(G) / G)
    elif kind == 1:
        s = np.zeros(G, np.int64)
        s[rng.integers(0, G)] = int(M * rng.uniform(0.7, 1.0))
    elif kind == 2:
        p = 1.0 / np.arange(1, G + 1) ** 1.2
        rng.shuffle(p)
        s = rng.multinomial(int(M * rng.uniform(0.8, 1.0)), p / p.sum())
    elif kind == 3:
        s = np.zeros(G, np.int64)
        idx = rng.choice(G, size=max(1, G // 4), replace=False)
        s[idx] = np.minimum(rng.integers(1, 40, size=idx.size), M // idx.size)
    else:
        s = rng.choice([16, 64, 128, 256], size=G) * rng.integers(0, 3, size=G) + rng.integers(-1, 2, size=G)
        s = np.maximum(s, 0)
    s = s.astype(np.int64)
    while s.sum() > M:  # trim the largest group until the rows fit
        j = int(np.argmax(s))
        s[j] -= min(s[j], s.sum() - M)
    return s.astype(np.int32)


def _deq_e4m3(q, scale_rows_cols):
    return q.view(torch.float8_e4m3fn).float() * scale_rows_cols


def _grouped_ref(a, w, off):
    """out[rows of g] = a[rows of g] @ w[g]^T (fp32), zero elsewhere."""
    out = torch.zeros(a.shape[0], w.shape[1], device=a.device)
    for g in range(w.shape[0]):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi > lo:
            out[lo:hi] = a[lo:hi] @ w[g].t()
    return out


def _within_fp8_bound(got, ref):
    return int(((got.float() - ref).abs() > 2e-3 + 1.5e-2 * ref.abs()).sum().item())


@pytest.mark.parametrize("seed", [101, 102, 103, 104])
def test_random_sweep(seed):
    rng = np.random.default_rng(seed)
    gen = torch.Generator(device="cuda").manual_seed(seed)
    dev = torch.device("cuda")
    for case in range(20):
        G = int(rng.choice([1, 2, 3, 8, 17, 64, 256]))
        M = int(rng.choice([1, 100, 513, 1024, 3000, 8192, 20000]))
        K = int(rng.choice([128, 256, 512, 1024, 2048]))
        N = int(rng.choice([128, 256, 384, 512]))
        fuse = bool(rng.integers(0, 2))
        s_np = _sizes(rng, G, M)
        S = int(s_np.sum())
        off = np.concatenate([[0], np.cumsum(s_np.astype(np.int64))])
        tag = f"seed {seed} case {case}: G={G} M={M} K={K} N={N} fuse={fuse} S={S}"
        s = torch.from_numpy(s_np).to(dev)
        Nw = 2 * N if fuse else N
        x = torch.randn(M, K, device=dev, generator=gen).to(torch.bfloat16)
        w = (torch.randn(G, K, Nw, device=dev, generator=gen) / math.sqrt(K)).to(torch.bfloat16)
        xq, xs = gmm.quantize_lhs(x)
        wq, ws = gmm.quantize_rhs(w)
        work = gmm.Workspace(G, M)

        # FP8 forward: configurations bit for bit, dequantized fp32 reference
        xd = _deq_e4m3(xq, xs.t().repeat_interleave(128, 1))
        wd = torch.stack([_deq_e4m3(wq[g], ws[g].t().repeat_interleave(128, 0).repeat_interleave(128, 1))
                          for g in range(G)])
        ref = _grouped_ref(xd, wd, off)
        if fuse:
            ref = torch.nn.functional.silu(ref[:, :N]) * ref[:, N:]
        cfgs = [None, (0, 5, 2, 1)]
        if fuse or N % 256 == 0:
            cfgs.append((0, 0, 0, 2))
        if not fuse and N % 256 == 0:
            cfgs.append((128, 0, 0, 1))
        outs = [gmm.fp8_fwd(xq, xs, wq, ws, s, fuse=fuse, workspace=work, config=c) for c in cfgs]
        torch.cuda.synchronize()
        assert work.status() == 0, tag
        for c, o in zip(cfgs[1:], outs[1:]):
            assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16)), f"{tag}: config {c} bits differ"
        assert _within_fp8_bound(outs[0], ref) == 0, f"{tag}: FP8 forward outside the bound"
        assert bool(torch.all(outs[0][S:] == 0).item()), f"{tag}: rows past the groups not zero"

        if fuse:
            h, hq, hs = gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, s, workspace=work)
            rq, rs = gmm.quantize_lhs(h)
            torch.cuda.synchronize()
            assert work.status() == 0, tag
            assert torch.equal(h.view(torch.int16), outs[0].view(torch.int16)), f"{tag}: h differs"
            assert torch.equal(hq, rq) and torch.equal(hs.view(torch.int32), rs.view(torch.int32)), f"{tag}: cast"

        # 4-bit weights
        wq4, ws4 = gmm.quantize_rhs_w4(w)
        lut = torch.tensor(E2M1, device=dev)
        codes = torch.stack([wq4 & 0xF, wq4 >> 4], dim=-1).reshape(G, Nw, K).long()
        wd4 = lut[codes] * ws4.transpose(1, 2).repeat_interleave(128, 1).repeat_interleave(128, 2)
        ref4 = _grouped_ref(xd, wd4, off)
        if fuse:
            ref4 = torch.nn.functional.silu(ref4[:, :N]) * ref4[:, N:]
        o4 = gmm.fp8_w4_fwd(xq, xs, wq4, ws4, s, fuse=fuse, workspace=work)
        if fuse or N % 256 == 0:
            o4p = gmm.fp8_w4_fwd(xq, xs, wq4, ws4, s, fuse=fuse, workspace=work, config=(0, 0, 0, 2))
            torch.cuda.synchronize()
            assert torch.equal(o4.view(torch.int16), o4p.view(torch.int16)), f"{tag}: 4-bit pair bits differ"
        torch.cuda.synchronize()
        assert work.status() == 0, tag
        assert _within_fp8_bound(o4, ref4) == 0, f"{tag}: 4-bit forward outside the bound"

        # tgmm
        Nt = int(rng.choice([128, 256, 512]))
        dy = torch.randn(M, Nt, device=dev, generator=gen).to(torch.bfloat16)
        d1 = gmm.tgmm(x, dy, s, workspace=work)
        d2 = gmm.tgmm(x, dy, s, workspace=work)
        torch.cuda.synchronize()
        assert work.status() == 0, tag
        assert torch.equal(d1.view(torch.int16), d2.view(torch.int16)), f"{tag}: tgmm not deterministic"
        refd = torch.zeros(G, K, Nt, device=dev)
        for g in range(G):
            lo, hi = int(off[g]), int(off[g + 1])
            if hi > lo:
                refd[g] = x[lo:hi].float().t() @ dy[lo:hi].float()
        # bf16 output rounding plus fp32 accumulation-order differences
        tol = 1e-2 * refd.abs() + 1e-2 + 1e-3 * math.sqrt(max(1, int(s_np.max())))
        assert int(((d1.float() - refd).abs() > tol).sum().item()) == 0, f"{tag}: tgmm outside the bound"

"""GPU parity of tgmm (dW[g] = X_g^T dY_g, bf16) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import make_case, normal_bf16
from tests.gpu_util import (BF16_ATOL, BF16_RTOL, Guarded, assert_close, bf16_to_np64, poison_bf16, to_dev,
                            to_dev_bf16)

pytestmark = pytest.mark.gpu

EDGE = [
    ([512], 512, 256, 256),
    ([0, 300, 0, 212], 512, 128, 256),
    ([1, 63, 64, 65, 0, 127, 128, 129], 700, 256, 384),
    ([5, 0, 0, 9], 20, 384, 128),
    ([0, 0, 0], 64, 128, 128),
    ([0, 0], 0, 128, 256),
    # K a multiple of 256: the CTA-pair kernel (256 k rows per pair of CTAs)
    ([3, 0, 200, 77], 300, 512, 256),
    ([130, 0, 150], 300, 768, 128),
    ([0, 0], 0, 256, 256),
]


@pytest.mark.parametrize("sizes,M,K,N", EDGE)
def test_tgmm_edges(sizes, M, K, N):
    rng = np.random.default_rng(M + K + N)
    s = np.array(sizes, np.int32)
    G = len(sizes)
    x = normal_bf16((M, K), 1.0, rng)
    dy = normal_bf16((M, N), 1.0, rng)
    dwg = Guarded((G, K, N), torch.bfloat16)
    work = gmm.Workspace(G, M)
    xt = to_dev_bf16(x) if M else torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    dyt = to_dev_bf16(dy) if M else torch.empty((0, N), dtype=torch.bfloat16, device="cuda")
    gmm.tgmm(xt, dyt, to_dev(s), dw=dwg.t, workspace=work)
    torch.cuda.synchronize()
    assert work.status() == 0
    dwg.check("tgmm dW")
    ref = oracle.tgmm_bf16(x, dy, s)
    got = bf16_to_np64(dwg.t)
    assert_close(got, ref, BF16_ATOL, BF16_RTOL, "tgmm")
    for g in range(G):
        if sizes[g] == 0:
            assert np.all(got[g] == 0)


def test_tgmm_dev_shape_full():
    c = make_case("tgmm_dev_bf16")
    dw = gmm.tgmm(to_dev_bf16(c.x), to_dev_bf16(c.dy), to_dev(c.group_sizes))
    torch.cuda.synchronize()
    ref = oracle.tgmm_bf16(c.x, c.dy, c.group_sizes)
    assert_close(bf16_to_np64(dw), ref, BF16_ATOL, BF16_RTOL, "tgmm dev")


def test_tgmm_many_small_groups():
    """4096 groups (the largest G), most of them empty or a few rows long, a
    few large: thousands of units, most with one partial chunk, which the
    CTA pairs claim several at a time; every dW[g] against the oracle and the
    empty groups' tiles zero."""
    rng = np.random.default_rng(4096)
    G, K, N = 4096, 256, 128  # the CTA-pair kernel with 128-column units
    sizes = np.where(rng.random(G) < 0.5, 0, rng.integers(1, 9, G)).astype(np.int32)
    sizes[[7, 1000, 4095]] = [700, 130, 64]
    M = int(sizes.sum()) + 5
    x = normal_bf16((M, K), 1.0, rng)
    dy = normal_bf16((M, N), 1.0, rng)
    dwg = Guarded((G, K, N), torch.bfloat16)
    dw = dwg.t
    work = gmm.Workspace(G, M)
    gmm.tgmm(to_dev_bf16(x), to_dev_bf16(dy), to_dev(sizes), dw=dw, workspace=work)
    torch.cuda.synchronize()
    assert work.status() == 0
    dwg.check("tgmm dW, 4096 groups")
    assert work.buf[16:24].view(torch.int32).tolist() == [0, 0]  # work counters back at zero
    got = bf16_to_np64(dw)
    ref = oracle.tgmm_bf16(x, dy, sizes)
    assert_close(got, ref, BF16_ATOL, BF16_RTOL, "tgmm, 4096 groups")
    assert np.all(got[sizes == 0] == 0)

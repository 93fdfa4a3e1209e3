"""GPU parity of the bf16 dgrad (dX_g = dY_g W[g]^T) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import make_case, normal_bf16
from tests.gpu_util import BF16_ATOL, BF16_RTOL, assert_close, bf16_to_np64, poison_bf16, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

EDGE = [
    ([512], 512, 256, 256),
    ([0, 300, 0, 212], 512, 384, 128),
    ([1, 127, 128, 129, 0, 2], 400, 256, 384),
    ([5, 0, 0, 9], 20, 128, 256),
    ([0, 0, 0], 64, 256, 128),
]


@pytest.mark.parametrize("sizes,M,K,N", EDGE)
def test_dgrad_edges(sizes, M, K, N):
    rng = np.random.default_rng(M + 3 * K + N)
    s = np.array(sizes, np.int32)
    G = len(sizes)
    dy = normal_bf16((M, N), 1.0, rng)
    w = normal_bf16((G, K, N), 1.0 / np.sqrt(N), rng)
    dx = poison_bf16(torch.empty((M, K), dtype=torch.bfloat16, device="cuda"))
    work = gmm.Workspace(G, M)
    gmm.dgrad(to_dev_bf16(dy), to_dev_bf16(w), to_dev(s), dx=dx, workspace=work)
    torch.cuda.synchronize()
    assert work.status() == 0
    ref = oracle.dgrad_bf16(dy, w, s)
    got = bf16_to_np64(dx)
    assert_close(got, ref, BF16_ATOL, BF16_RTOL, "dgrad")
    assert np.all(got[int(s.sum()):] == 0)


def test_dgrad_dev_shape_full():
    # the wi layer's dgrad at the development shape: dY [8192, 512], W [32, 2048, 512]
    c = make_case("wi_dev_fp8")
    rng = np.random.default_rng(77)
    dy = normal_bf16((c.M, c.N), 1.0, rng)
    dx = gmm.dgrad(to_dev_bf16(dy), to_dev_bf16(c.w), to_dev(c.group_sizes))
    torch.cuda.synchronize()
    ref = oracle.dgrad_bf16(dy, c.w, c.group_sizes)
    assert_close(bf16_to_np64(dx), ref, BF16_ATOL, BF16_RTOL, "dgrad dev")

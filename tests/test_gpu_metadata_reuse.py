"""group_sizes = NULL: a grouped call reuses the group metadata already in its
workspace (written by gmm_group_metadata, or by an earlier grouped call with
the same G and M on the same stream).  Every grouped entry point must then
give bit for bit what it gives when it derives the metadata itself."""
import numpy as np
import pytest
import torch

import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import normal_bf16
from tests.gpu_util import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sizes,M,K,N", [([0, 300, 0, 212], 512, 256, 256), ([77, 1, 0, 130, 5], 300, 512, 384)])
def test_null_group_sizes_reuses_metadata(sizes, M, K, N):
    rng = np.random.default_rng(7 + M)
    G = len(sizes)
    s = to_dev(np.array(sizes, np.int32))
    x = to_dev_bf16(normal_bf16((M, K), 1.0, rng))
    w = to_dev_bf16(normal_bf16((G, K, 2 * N), 1.0 / np.sqrt(K), rng))
    w1 = w[:, :, :N].contiguous()
    dy = to_dev_bf16(normal_bf16((M, N), 1.0, rng))
    xq, xs = gmm.quantize_lhs(x)
    wq, ws = gmm.quantize_rhs(w)
    wq1, ws1 = gmm.quantize_rhs(w1)

    ref = [gmm.fp8_fwd(xq, xs, wq1, ws1, s), gmm.fp8_fwd(xq, xs, wq, ws, s, fuse=True),
           *gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, s), gmm.bf16_fwd(x, w1, s), gmm.dgrad(dy, w1, s),
           gmm.tgmm(x, dy, s)]

    work = gmm.group_metadata(s, M)
    got = [gmm.fp8_fwd(xq, xs, wq1, ws1, None, workspace=work),
           gmm.fp8_fwd(xq, xs, wq, ws, None, fuse=True, workspace=work),
           *gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, None, workspace=work),
           gmm.bf16_fwd(x, w1, None, workspace=work), gmm.dgrad(dy, w1, None, workspace=work),
           gmm.tgmm(x, dy, None, workspace=work)]
    torch.cuda.synchronize()
    assert work.status() == 0
    for i, (a, b) in enumerate(zip(ref, got)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"output {i} differs"


def test_null_group_sizes_needs_a_workspace():
    xq = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    xs = torch.zeros((1, 128), dtype=torch.float32, device="cuda")
    wq = torch.zeros((2, 128, 128), dtype=torch.uint8, device="cuda")
    ws = torch.zeros((2, 1, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        gmm.fp8_fwd(xq, xs, wq, ws, None)


def test_tgmm_work_counters_return_to_zero():
    """The CTA-pair tgmm claims its units from two workspace words (units
    claimed, CTAs finished); each launch must leave them at zero, so that
    back-to-back calls on one workspace, of different shapes, each see every
    unit once and give the same bits as a call that ran its own metadata."""
    rng = np.random.default_rng(11)
    sizes = [700, 0, 3, 260, 129, 64, 1, 0, 900, 17]
    G, M = len(sizes), sum(sizes) + 37
    s = to_dev(np.array(sizes, np.int32))
    shapes = [(512, 512), (256, 256), (512, 1024)]
    data = []
    for K, N in shapes:
        x = to_dev_bf16(normal_bf16((M, K), 1.0, rng))
        dy = to_dev_bf16(normal_bf16((M, N), 1.0, rng))
        data.append((x, dy, gmm.tgmm(x, dy, s)))
    work = gmm.group_metadata(s, M)
    for _ in range(3):
        for x, dy, ref in data:
            got = gmm.tgmm(x, dy, None, workspace=work)
            assert torch.equal(ref.view(torch.uint8), got.view(torch.uint8))
    torch.cuda.synchronize()
    assert work.status() == 0
    assert work.buf[16:24].view(torch.int32).tolist() == [0, 0]  # words 4 and 5

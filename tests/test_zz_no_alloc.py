"""gmm_fp8_fwd_noalloc: the FP8 grouped forward for callers that cannot
allocate device memory when they run the layer.

Such callers exist: code running under a framework whose caching allocator
owns all device memory, runtimes that must not allocate after start-up (fixed
memory budgets, real-time serving loops), and plug-ins that are handed only
their input and output buffers.  They cannot provide the workspace that
gmm_fp8_fwd takes, so this entry point keeps its group metadata in a fixed
64 KiB array in the library's own device memory.

The test calls the entry point through the C ABI twice in a row, with
different group layouts (the second call must not see the first call's
metadata), and checks each output against gmm_fp8_fwd with a workspace bit
for bit: both run the same kernel with the same tile configuration.  This file is collected
last on purpose; it passes on its own in a fresh process as well.
"""
import numpy as np
import pytest
import torch

import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import normal_bf16
from tests.gpu_util import poison_bf16, to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def _case(sizes, M, K, N, fuse, seed):
    rng = np.random.default_rng(seed)
    G = len(sizes)
    x = normal_bf16((M, K), 1.0, rng, outlier_p=0.01)
    w = normal_bf16((G, K, 2 * N if fuse else N), 1.0 / np.sqrt(K), rng)
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    wq, ws = gmm.quantize_rhs(to_dev_bf16(w))
    return dict(xq=xq, xs=xs, wq=wq, ws=ws, sizes=to_dev(np.array(sizes, np.int32)), G=G, M=M, K=K, N=N,
                fuse=fuse)


def _with_workspace(c):
    return gmm.fp8_fwd(c["xq"], c["xs"], c["wq"], c["ws"], c["sizes"], fuse=c["fuse"])


def _no_alloc(c):
    out = poison_bf16(torch.empty((c["M"], c["N"]), dtype=torch.bfloat16, device="cuda"))
    st = gmm.gmm_fp8_fwd_noalloc(c["xq"], c["xs"], c["wq"], c["ws"], c["sizes"], c["G"], c["M"], c["K"], c["N"],
                                 c["fuse"], out)
    assert st == 0, gmm.STATUS_NAMES.get(st, st)
    return out


def test_no_alloc_matches_workspace_entry_point_twice_in_a_row():
    first = _case([300, 0, 129, 1, 270], 760, 512, 512, False, 11)
    second = _case([5, 640, 0], 700, 256, 384, True, 12)
    got1 = _no_alloc(first)
    got2 = _no_alloc(second)
    torch.cuda.synchronize()
    ref1 = _with_workspace(first)
    ref2 = _with_workspace(second)
    torch.cuda.synchronize()
    # the same kernel with the same tile configuration on the same inputs:
    # every element must carry the same bits
    assert torch.equal(got1.view(torch.int16), ref1.view(torch.int16)), "no-alloc call 1 differs from gmm_fp8_fwd"
    assert torch.equal(got2.view(torch.int16), ref2.view(torch.int16)), "no-alloc call 2 differs from gmm_fp8_fwd"
    # rows past sum(group_sizes) are zero in both
    assert torch.all(got1[700:] == 0) and torch.all(got2[645:] == 0)


def test_no_alloc_refuses_sizes_beyond_its_scratch():
    # 4096 groups x 2^20 rows need far more than the 64 KiB static array
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    st = gmm.gmm_fp8_fwd_noalloc(dummy, dummy, dummy, dummy, dummy, 4096, 1 << 20, 128, 128, 0, dummy)
    assert st == 8  # GMM_ERR_WORKSPACE, nothing launched

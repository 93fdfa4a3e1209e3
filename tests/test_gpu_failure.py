"""Failure detection on the GPU without a fault: a wait that nothing completes
ends in a status the host reads, and the context stays usable afterwards."""
import time

import numpy as np
import pytest
import torch

import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import normal_bf16
from tests.gpu_util import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu


def test_stuck_wait_reports_timeout_and_context_survives():
    work = gmm.Workspace(1, 1)
    t0 = time.perf_counter()
    assert gmm.gmm_selftest_wait_timeout(work.buf, work.nbytes, 200) == 0
    assert gmm.gmm_get_device_status(work.buf) == 7  # GMM_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    # the short wait gives up after ~0.2 s and the other warps (2 s limit)
    # stop through the abort word instead of running out their own limit
    assert 0.15 < elapsed < 1.5, elapsed
    assert gmm.gmm_get_device_status(work.buf) == 0  # read-and-clear

    # the same process still runs the real kernels correctly
    rng = np.random.default_rng(3)
    x = normal_bf16((256, 256), 1.0, rng)
    w = normal_bf16((2, 256, 256), 1.0 / 16, rng)
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    wq, ws = gmm.quantize_rhs(to_dev_bf16(w))
    sizes = to_dev(np.array([100, 156], np.int32))
    a = gmm.fp8_fwd(xq, xs, wq, ws, sizes, workspace=work)
    b = gmm.bf16_fwd(to_dev_bf16(x), to_dev_bf16(w), sizes, workspace=work)
    torch.cuda.synchronize()
    assert work.status() == 0
    rel = (a.float() - b.float()).norm() / b.float().norm()
    assert rel < 0.1


def test_selftest_validates_arguments():
    work = gmm.Workspace(1, 1)
    assert gmm.gmm_selftest_wait_timeout(work.buf, work.nbytes, 0) == 2
    assert gmm.gmm_selftest_wait_timeout(None, 0, 100) == 8

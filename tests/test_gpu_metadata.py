"""GPU parity of the device metadata kernel (group offsets, the 128-row and
256-row tile lists) against the oracle, bit-exact, and its error reporting."""
import numpy as np
import pytest
import torch

import oracle
import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import routing_sizes
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

CASES = [
    ([512], 512), ([0, 0, 0, 0], 100), ([0, 5, 0], 5), ([1, 127, 128, 129, 0, 256], 700),
    ([3, 0, 5], 20), ([128] * 64, 8192), (list(range(300)), 44850), ([0] * 4095 + [7], 7),
    ([1] * 4096, 4096), ([], 0),
]


@pytest.mark.parametrize("sizes,M", [c for c in CASES if c[0]] + [
    (routing_sizes("wi_dev_fp8").tolist(), 8192), (routing_sizes("prod_fp8").tolist(), 65536)])
def test_offsets_and_tiles(sizes, M):
    s = np.array(sizes, np.int32)
    ws = gmm.group_metadata(to_dev(s), M)
    torch.cuda.synchronize()
    off, tiles = oracle.group_tiles(s, M, 128)
    hdr = ws.header()
    assert hdr[0] == 0 and hdr[1] == 1
    assert hdr[2] == off[-1] and hdr[3] == len(tiles)
    assert ws.offsets() == off.tolist()
    assert np.array_equal(ws.tiles().cpu().numpy(), tiles.astype(np.int32))
    _, tiles2 = oracle.group_tiles(s, M, 256)
    assert ws.buf[24:28].view(torch.int32).item() == len(tiles2)
    assert np.array_equal(ws.pair_tiles().cpu().numpy(), tiles2.astype(np.int32))
    # the group ids by size, largest first, ties by id (numpy's stable sort)
    sz = np.asarray(sizes, np.int64)
    assert ws.order() == np.argsort(-sz, kind="stable").tolist()
    assert gmm.gmm_get_device_status(ws.buf) == 0


@pytest.mark.parametrize("sizes,M,want", [([3, -1, 2], 10, 6), ([5, 6], 10, 6), ([-5], 10, 6)])
def test_invalid_sizes_set_status(sizes, M, want):
    s = np.array(sizes, np.int32)
    ws = gmm.group_metadata(to_dev(s), M)
    torch.cuda.synchronize()
    hdr = ws.header()
    assert hdr[1] == 0 and hdr[3] == 0
    assert gmm.gmm_get_device_status(ws.buf) == want
    assert gmm.gmm_get_device_status(ws.buf) == 0  # read-and-clear


def test_invalid_sizes_leave_no_tiles_for_the_gemm():
    # an FP8 forward with bad sizes writes nothing and reports GMM_ERR_GROUP_SIZES
    G, M, K, N = 2, 256, 128, 128
    xq = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    xs = torch.ones((1, M), dtype=torch.float32, device="cuda")
    wq = torch.zeros((G, N, K), dtype=torch.uint8, device="cuda")
    wsc = torch.ones((G, 1, 1), dtype=torch.float32, device="cuda")
    out = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    work = gmm.Workspace(G, M)
    gmm.fp8_fwd(xq, xs, wq, wsc, to_dev(np.array([200, 100], np.int32)), out=out, workspace=work)
    assert work.status() == 6
    assert torch.all(out == 3.0)

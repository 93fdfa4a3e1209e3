"""GPU parity of the blockwise quantization kernels against the oracle:
e4m3 codes and fp32 scales must be bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300.workloads import f32_to_bf16_bits, make_case, normal_bf16
from tests.gpu_util import to_dev_bf16

pytestmark = pytest.mark.gpu


def _edge_rows(K, rng):
    """Rows whose blocks hit the quantizer's special cases."""
    rows = []
    z = np.zeros(K, np.float32)
    rows.append(z)                                            # all-zero blocks: scale 0
    neg0 = np.full(K, -0.0, np.float32)
    rows.append(neg0)                                         # -0.0 keeps its sign
    r = rng.standard_normal(K).astype(np.float32)
    r[::128] = 448.0                                          # absmax 448: scale 1
    rows.append(r)
    rows.append(np.ldexp(np.ones(K, np.float32), rng.integers(-30, 30, K)).astype(np.float32))
    rows.append((rng.standard_normal(K) * 1e-30).astype(np.float32))   # tiny but normal scales
    rows.append((rng.standard_normal(K) * 3e4).astype(np.float32))     # large
    one_hot = np.zeros(K, np.float32)
    one_hot[5] = -7.0
    rows.append(one_hot)                                      # a single non-zero per block
    ties = np.tile(np.array([1.0625, 1.1875, 17.0, 19.0, 448.0, -3 * 2.0 ** -10 * 448], np.float32),
                   K // 6 + 1)[:K]
    rows.append(ties)                                         # e4m3 rounding ties at scale 1
    return f32_to_bf16_bits(np.stack(rows))


@pytest.mark.parametrize("M,K", [(1, 128), (37, 384), (513, 256), (1000, 1024)])
def test_lhs_bit_exact_random_and_edges(M, K):
    rng = np.random.default_rng(M * 7 + K)
    x = normal_bf16((M, K), 1.0, rng, outlier_p=0.02)
    e = _edge_rows(K, rng)
    x[: min(M, len(e))] = e[: min(M, len(e))]
    xq, xs = gmm.quantize_lhs(to_dev_bf16(x))
    torch.cuda.synchronize()
    oxq, oxs = oracle.quantize_lhs(x)
    assert np.array_equal(xq.cpu().numpy(), oxq)
    assert np.array_equal(xs.cpu().numpy().T.view(np.uint32), oxs.view(np.uint32))


def test_lhs_bit_exact_dev_shape():
    c = make_case("wi_dev_fp8")
    xq, xs = gmm.quantize_lhs(to_dev_bf16(c.x))
    torch.cuda.synchronize()
    oxq, oxs = oracle.quantize_lhs(c.x)
    assert np.array_equal(xq.cpu().numpy(), oxq)
    assert np.array_equal(xs.cpu().numpy().T.view(np.uint32), oxs.view(np.uint32))


def test_lhs_empty_is_noop():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    xq, xs = gmm.quantize_lhs(x)
    assert xq.shape == (0, 256) and xs.shape == (2, 0)


@pytest.mark.parametrize("G,K,N", [(1, 128, 128), (3, 256, 384), (4, 512, 1024)])
def test_rhs_bit_exact(G, K, N):
    rng = np.random.default_rng(G * 100 + K + N)
    w = normal_bf16((G, K, N), 1.0 / np.sqrt(K), rng, outlier_p=0.01)
    w[0, :128, :128] = 0                                      # one all-zero block
    wq, ws = gmm.quantize_rhs(to_dev_bf16(w))
    torch.cuda.synchronize()
    owq, ows = oracle.quantize_rhs(w)
    # the library stores wq K-major: wq[g, n, k] is the code of w[g, k, n]
    assert np.array_equal(wq.cpu().numpy().transpose(0, 2, 1), owq)
    assert np.array_equal(ws.cpu().numpy().view(np.uint32), ows.view(np.uint32))

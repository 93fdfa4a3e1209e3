"""The tile configurations on the GPU: every configuration the autotuner may
choose (FP8 forward: bn, CTA count, unit order, CTA group, ring slots, TMEM
buffers; tgmm: ring slots, claim-ahead, claim batch) gives the default
configuration's bits (the same sums in the same order), on ragged cases with
empty groups, partial tiles and tail rows, plain, fused and with the fused
FP8 cast; the device-dependent configuration errors; and short autotuner runs
whose winners pass the gate.  The default configurations themselves are
checked against the oracle in test_gpu_gmm.py and test_gpu_tgmm.py."""
import numpy as np
import pytest
import torch

import fp8_blockwise_quantized_gb300 as gmm
from fp8_blockwise_quantized_gb300 import tune
from fp8_blockwise_quantized_gb300.workloads import normal_bf16
from tests.gpu_util import to_dev, to_dev_bf16

pytestmark = pytest.mark.gpu

CASES = [
    ([300, 0, 129, 1, 640], 1200, 512, 512),
    ([77, 300, 1, 255, 256, 33], 1000, 256, 768),
    ([0, 0, 0], 64, 256, 256),
]


def _problem(sizes, M, K, Nw, seed):
    rng = np.random.default_rng(seed)
    s = to_dev(np.array(sizes, np.int32))
    x = to_dev_bf16(normal_bf16((M, K), 1.0, rng, outlier_p=0.01))
    w = to_dev_bf16(normal_bf16((len(sizes), K, Nw), 1.0 / np.sqrt(K), rng))
    xq, xs = gmm.quantize_lhs(x)
    wq, ws = gmm.quantize_rhs(w)
    return s, xq, xs, wq, ws


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _even(n):
    return n - n % 2


@pytest.mark.parametrize("sizes,M,K,N", CASES)
def test_every_config_gives_the_default_bits(sizes, M, K, N):
    s, xq, xs, wq, ws = _problem(sizes, M, K, N, 5 + M)
    ref = gmm.fp8_fwd(xq, xs, wq, ws, s)
    sms = _sms()
    # every member of the autotuner's space (bn, CTA count, unit order, CTA
    # group, ring slots, TMEM buffers), plus a few small CTA counts
    cfgs = tune.fp8_space(N, False, sms).members()
    cfgs += [(128, c, 1, 1, 4, 2) for c in (1, 7)] + [(128, 3, 2, 1, 5, 4)]
    if N % 256 == 0:
        cfgs += [(256, 1, 1, 1, 3, 2), (256, 2, 2, 2, 3, 4), (256, 8, 1, 2, 4, 4)]
    for cfg in cfgs:
        got = gmm.fp8_fwd(xq, xs, wq, ws, s, config=cfg)
        assert torch.equal(ref.view(torch.int16), got.view(torch.int16)), cfg


def test_fused_configs_give_the_default_bits():
    sizes, M, K, N = [300, 0, 129, 1, 640], 1200, 512, 256
    s, xq, xs, wq, ws = _problem(sizes, M, K, 2 * N, 17)
    ref = gmm.fp8_fwd(xq, xs, wq, ws, s, fuse=True)
    for cfg in tune.fp8_space(N, True, _sms()).members() + [(256, 3, 1, 1, 2, 2), (256, 2, 2, 2, 5, 4)]:
        got = gmm.fp8_fwd(xq, xs, wq, ws, s, fuse=True, config=cfg)
        assert torch.equal(ref.view(torch.int16), got.view(torch.int16)), cfg


def test_tgmm_configs_give_the_default_bits():
    """Every ring depth, claim-ahead and claim batch of the CTA-pair tgmm
    kernel gives the default's dW bits (the same sums in the same order), on
    many small groups (batched claims), a large one and empty ones; the work
    counters are back at zero after every launch."""
    rng = np.random.default_rng(71)
    G, K, N = 300, 512, 256
    sizes = np.where(rng.random(G) < 0.3, 0, rng.integers(1, 40, G)).astype(np.int32)
    sizes[[3, 100]] = [900, 257]
    M = int(sizes.sum()) + 9
    x = to_dev_bf16(normal_bf16((M, K), 1.0, rng))
    dy = to_dev_bf16(normal_bf16((M, N), 1.0, rng))
    sd = to_dev(sizes)
    work = gmm.Workspace(G, M)
    ref = gmm.tgmm(x, dy, sd, workspace=work)
    for cfg in tune.tgmm_space(K, N).members():
        got = gmm.tgmm(x, dy, sd, workspace=work, config=cfg)
        torch.cuda.synchronize()
        assert torch.equal(ref.view(torch.int16), got.view(torch.int16)), cfg
        assert work.buf[16:24].view(torch.int32).tolist() == [0, 0], cfg
    assert work.status() == 0


def test_tgmm_autotuner_winner_passes_the_gate():
    rng = np.random.default_rng(72)
    sizes = np.array([700, 0, 3, 260, 129, 64, 1, 900], np.int32)
    M, K, N = int(sizes.sum()), 512, 512
    x = to_dev_bf16(normal_bf16((M, K), 1.0, rng))
    dy = to_dev_bf16(normal_bf16((M, N), 1.0, rng))
    r = tune.tune_tgmm(x, dy, to_dev(sizes), generations=2, population=4, reps=2, seed=3)
    assert tune.tgmm_space(K, N).contains(r.best) and r.default == (6, 3, 4)
    assert all(ok for _, _, _, ok in r.history)


def test_config_errors_on_the_device():
    s, xq, xs, wq, ws = _problem([100, 28], 128, 256, 384, 3)
    # N = 384: no 256-column units (bn 256, CTA pairs); bad counts and values
    for cfg in [(256, 0, 1), (0, _sms() + 1, 1), (64, 0, 1), (0, 0, 3), (0, 0, 1, 2), (0, 0, 1, 3)]:
        with pytest.raises(gmm.GmmError) as e:
            gmm.fp8_fwd(xq, xs, wq, ws, s, config=cfg)
        assert e.value.status == 4, cfg
    # the fused gate/up weight (2N = 512 columns) has 256-column units only
    s, xq, xs, wq, ws = _problem([100, 28], 128, 256, 512, 4)
    with pytest.raises(gmm.GmmError) as e:
        gmm.fp8_fwd(xq, xs, wq, ws, s, fuse=True, config=(128, 0, 1))
    assert e.value.status == 4
    # CTA pairs need an even CTA count
    with pytest.raises(gmm.GmmError) as e:
        gmm.fp8_fwd(xq, xs, wq, ws, s, fuse=True, config=(256, 7, 1, 2))
    assert e.value.status == 4


def test_autotuner_winner_passes_the_gate():
    sizes, M, K, N = [700, 0, 3, 260, 129, 64, 1, 900], 2100, 512, 512
    s, xq, xs, wq, ws = _problem(sizes, M, K, N, 23)
    r = tune.tune_fp8_fwd(xq, xs, wq, ws, s, generations=2, population=4, reps=2, seed=1)
    sp = tune.fp8_space(N, False, _sms())
    assert sp.contains(r.best) and r.default == tune.default_config(sp)
    assert all(ok for _, _, _, ok in r.history)  # every configuration gives the default's bits
    ref = gmm.fp8_fwd(xq, xs, wq, ws, s)
    got = gmm.fp8_fwd(xq, xs, wq, ws, s, config=r.best)
    assert torch.equal(ref.view(torch.int16), got.view(torch.int16))
    assert r.best_ms <= r.default_ms


def test_fused_cast_configs_give_the_default_bits():
    """The wi launch that also writes h's FP8 cast: h, the e4m3 codes and the
    scales of every configuration equal the default's."""
    sizes, M, K, N = [300, 0, 129, 1, 640], 1200, 512, 256
    s, xq, xs, wq, ws = _problem(sizes, M, K, 2 * N, 29)
    ref = gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, s)
    for cfg in tune.fp8_space(N, True, _sms()).members() + [(256, 5, 1, 1, 2, 2), (256, 4, 2, 2, 3, 4)]:
        got = gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, s, config=cfg)
        for a, b in zip(ref, got):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), cfg
    with pytest.raises(gmm.GmmError) as e:
        gmm.fp8_fwd_swiglu_quant(xq, xs, wq, ws, s, config=(128, 0, 1))
    assert e.value.status == 4


def test_autotuner_on_the_fused_cast_launch():
    sizes, M, K, N = [700, 0, 3, 260, 129, 64, 1, 900], 2100, 512, 256
    s, xq, xs, wq, ws = _problem(sizes, M, K, 2 * N, 31)
    r = tune.tune_fp8_fwd(xq, xs, wq, ws, s, quant=True, generations=2, population=3, reps=2, seed=2)
    assert r.best[0] == 256 and all(ok for _, _, _, ok in r.history)

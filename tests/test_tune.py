"""Host logic of the tile autotuner: the FP8 and tgmm search spaces (the
library's own rules for which combinations exist), mutation with repair, and
the evolutionary selection with its accuracy gate (a synthetic evaluator
stands in for the GPU timings; tests/test_gpu_tune.py runs it on the device)."""
import random

import pytest

from fp8_blockwise_quantized_gb300 import tune


def test_fp8_space_follows_the_library_rules():
    sp = tune.fp8_space(512, False, 152)
    assert sp.values[0] == (128, 256) and sp.values[3] == (1, 2)
    assert sp.values[1] == (76, 94, 114, 132, 152)  # even CTA counts, so CTA pairs can use each
    assert tune.fp8_space(384, False, 152).values[0] == (128,)   # 256 needs N % 256 == 0
    assert tune.fp8_space(384, False, 152).values[3] == (1,)     # and so do CTA pairs
    assert tune.fp8_space(512, True, 152).values[0] == (256,)    # fused units are 256 columns of W
    assert sp.default == (256, 152, 1, 1, 3, 2) and sp.contains(sp.default)
    assert tune.fp8_space(384, False, 8).default == (128, 8, 1, 1, 4, 2)
    # the compiled instances: bn 256 rings of 2-3 slots and 2 TMEM buffers; bn
    # 128 rings of 3-5 slots and 2 or 4 buffers; pairs 256-column units, 4
    # buffers, 3-4 slots (3-5 fused)
    assert sp.contains((128, 152, 1, 1, 5, 4)) and not sp.contains((128, 152, 1, 1, 2, 2))
    assert not sp.contains((256, 152, 1, 1, 4, 2)) and not sp.contains((256, 152, 1, 1, 3, 4))
    assert sp.contains((256, 152, 2, 2, 4, 4)) and not sp.contains((256, 152, 1, 2, 5, 4))
    assert tune.fp8_space(512, True, 152).contains((256, 152, 1, 2, 5, 4))
    assert not sp.contains((128, 152, 1, 2, 4, 4))
    assert all(sp.valid(c) for c in sp.members()) and len(sp.members()) == 100


def test_tgmm_space():
    sp = tune.tgmm_space(2048, 1024)
    assert sp.names == ("stages", "claim_ahead", "max_batch") and sp.default == (6, 3, 4)
    assert sp.values[0] == (4, 5, 6) and sp.contains((4, 8, 1))
    assert tune.tgmm_space(2048, 384).values[0] == (6,)  # 128-column units: the ring is fixed


def test_mutation_moves_one_field_and_repairs_the_rest():
    sp = tune.fp8_space(512, False, 152)
    rng = random.Random(3)
    c = sp.default
    for _ in range(300):
        m = tune.mutate(c, sp, rng)
        assert sp.contains(m) and m != c
        # some field moved to a neighbouring value; any other change was
        # forced by the rule
        moved = [i for i in range(len(c)) if m[i] != c[i]]
        assert any(abs(sp.values[i].index(m[i]) - sp.values[i].index(c[i])) == 1 for i in moved)
        c = m
    # CTA pairs are reachable from the default in one mutation (repairing the
    # TMEM buffer count)
    seen = {tune.mutate(sp.default, sp, random.Random(s)) for s in range(200)}
    assert any(m[3] == 2 for m in seen)


def _cost(c):
    # a synthetic landscape over (bn, ctas, order, cta_group, stages, bufs)
    # with its minimum at (128, 114, 2, 1, 5, 4)
    return (abs(c[0] - 128) / 64 + abs(c[1] - 114) / 19 + (0 if c[2] == 2 else 1.5) + (0 if c[3] == 1 else 2)
            + abs(c[4] - 5) / 2 + (0 if c[5] == 4 else 1) + 1.0)


def test_evolve_finds_the_optimum_and_measures_each_config_once():
    sp = tune.fp8_space(512, False, 152)
    calls = []

    def evaluate(c):
        calls.append(c)
        return _cost(c), True

    r = tune.evolve(evaluate, sp, generations=12, population=8, seed=1)
    assert r.best == (128, 114, 2, 1, 5, 4)
    assert r.default == sp.default and r.default_ms == _cost(sp.default)
    assert len(calls) == len(set(calls))
    assert all(sp.contains(c) for c in calls)


def test_gate_rejects_faster_wrong_configs():
    sp = tune.fp8_space(512, False, 152)

    def evaluate(c):
        wrong = c[2] == 2          # pretend column-major gives different bits
        return _cost(c) - (5 if wrong else 0), not wrong

    r = tune.evolve(evaluate, sp, generations=8, population=6, seed=2)
    assert r.best[2] == 1
    assert all(ok or c[2] == 2 for _, c, _, ok in r.history)


def test_no_passing_config_is_an_error():
    sp = tune.fp8_space(512, False, 152)
    with pytest.raises(RuntimeError):
        tune.evolve(lambda c: (1.0, False), sp, generations=2, population=3)


def test_evolve_is_deterministic_for_a_seed():
    sp = tune.tgmm_space(2048, 1024)
    cost = lambda c: abs(c[0] - 5) + abs(c[1] - 4) / 2 + abs(c[2] - 2)
    a = tune.evolve(lambda c: (cost(c), True), sp, generations=3, population=5, seed=9)
    b = tune.evolve(lambda c: (cost(c), True), sp, generations=3, population=5, seed=9)
    assert a.history == b.history


def test_a_timed_out_candidate_fails_the_gate():
    from fp8_blockwise_quantized_gb300 import binding
    assert tune.status_passes(binding.GMM_OK)
    # a bounded wait ran out: the launch stopped early and its time is no
    # measurement, so the candidate fails (and never becomes a parent)
    assert not tune.status_passes(binding.GMM_ERR_TIMEOUT)
    with pytest.raises(RuntimeError):
        tune.status_passes(binding.GMM_ERR_GROUP_SIZES, "config (256, 152, 1, 1, 3, 2)")

"""Host logic of the FP8 tile autotuner: the search space, mutation, and the
evolutionary selection with its accuracy gate (a synthetic evaluator stands
in for the GPU timings; tests/test_gpu_tune.py runs it on the device)."""
import random

import pytest

from fp8_blockwise_quantized_gb300 import tune


def test_space_follows_the_library_rules():
    assert tune.space_for(512, False, 152).bns == (128, 256)
    assert tune.space_for(384, False, 152).bns == (128,)   # 256 needs N % 256 == 0
    assert tune.space_for(512, True, 152).bns == (256,)    # fused units are 256 columns of W
    sp = tune.space_for(512, False, 152)
    assert sp.ctas == (76, 95, 114, 133, 152) and max(sp.ctas) == 152
    assert tune.default_config(sp) == (256, 152, 1)
    assert tune.default_config(tune.space_for(384, False, 8)) == (128, 8, 1)


def test_mutation_changes_one_field_to_a_neighbour():
    sp = tune.space_for(512, False, 152)
    rng = random.Random(3)
    c = (256, 114, 1)
    for _ in range(200):
        m = tune.mutate(c, sp, rng)
        assert sp.contains(m) and m != c
        diff = [i for i in range(3) if m[i] != c[i]]
        assert len(diff) == 1
        vals = (sp.bns, sp.ctas, sp.orders)[diff[0]]
        assert abs(vals.index(m[diff[0]]) - vals.index(c[diff[0]])) == 1
        c = m


def _cost(c):
    # a synthetic landscape with its minimum at (256, 114, 2)
    return abs(c[0] - 256) / 64 + abs(c[1] - 114) / 19 + (0 if c[2] == 2 else 1.5) + 1.0


def test_evolve_finds_the_optimum_and_measures_each_config_once():
    sp = tune.space_for(512, False, 152)
    calls = []

    def evaluate(c):
        calls.append(c)
        return _cost(c), True

    r = tune.evolve(evaluate, sp, generations=8, population=6, seed=1)
    assert r.best == (256, 114, 2)
    assert r.default == (256, 152, 1) and r.default_ms == _cost((256, 152, 1))
    assert len(calls) == len(set(calls))
    assert all(sp.contains(c) for c in calls)


def test_gate_rejects_faster_wrong_configs():
    sp = tune.space_for(512, False, 152)

    def evaluate(c):
        wrong = c[2] == 2          # pretend column-major gives different bits
        return _cost(c) - (5 if wrong else 0), not wrong

    r = tune.evolve(evaluate, sp, generations=8, population=6, seed=2)
    assert r.best[2] == 1
    assert all(ok or c[2] == 2 for _, c, _, ok in r.history)


def test_no_passing_config_is_an_error():
    sp = tune.space_for(512, False, 152)
    with pytest.raises(RuntimeError):
        tune.evolve(lambda c: (1.0, False), sp, generations=2, population=3)


def test_evolve_is_deterministic_for_a_seed():
    sp = tune.space_for(512, False, 152)
    a = tune.evolve(lambda c: (_cost(c), True), sp, generations=3, population=5, seed=9)
    b = tune.evolve(lambda c: (_cost(c), True), sp, generations=3, population=5, seed=9)
    assert a.history == b.history


def test_a_timed_out_candidate_fails_the_gate():
    from fp8_blockwise_quantized_gb300 import binding
    assert tune.status_passes(binding.GMM_OK)
    # a bounded wait ran out: the launch stopped early and its time is no
    # measurement, so the candidate fails (and never becomes a parent)
    assert not tune.status_passes(binding.GMM_ERR_TIMEOUT)
    with pytest.raises(RuntimeError):
        tune.status_passes(binding.GMM_ERR_GROUP_SIZES, "config (256, 152, 1)")

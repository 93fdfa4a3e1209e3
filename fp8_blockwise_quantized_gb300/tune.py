"""Tile autotuner for the FP8 forward.

The search follows "GEMM Kernel 性能优化十问", Q8 and Q9.4.  Tile sizes are
chosen by a search over candidates measured on the real shapes. A candidate
may win only after an accuracy check, which a caller can loosen but never
switch off.

The space is the library's ``gmm_fp8_tile_config``:
- ``bn``: the MMA N of a work unit, 128 or 256;
- ``ctas``: the number of persistent CTAs;
- ``unit_order``: the order of the work units, 1 row-tile major, 2 column-block major.

The search is evolutionary. The first population holds the default and random
members. Each generation keeps the fastest members that pass the gate and
fills up with mutants of them; a mutant has one field moved to a neighbouring
value.

The gate compares a candidate's output with the output of the default
configuration. The test is bit for bit, since every configuration computes
the same sums in the same order. A caller may loosen it to an atol/rtol bound.

Timing uses CUDA events on the launching stream, after one untimed run, with
L2 flushed between runs. Everything measured runs in the library's kernels;
this module only chooses arguments.
"""
from __future__ import annotations

import random
from dataclasses import dataclass, field

import torch

from . import binding

Config = tuple  # (bn, ctas, unit_order)


@dataclass(frozen=True)
class Space:
    """The configurations a shape admits."""
    bns: tuple
    ctas: tuple
    orders: tuple = (1, 2)

    def contains(self, c: Config) -> bool:
        return c[0] in self.bns and c[1] in self.ctas and c[2] in self.orders


def space_for(N: int, fuse: bool, sms: int) -> Space:
    """bn 256 needs N % 256 == 0 and is the only value for the fused gate/up
    weight; the CTA counts are the SM count and fractions of it."""
    bns = (256,) if fuse else ((128, 256) if N % 256 == 0 else (128,))
    ctas = tuple(sorted({max(1, sms * f // 8) for f in (4, 5, 6, 7, 8)}))
    return Space(bns, ctas)


def default_config(space: Space) -> Config:
    return (max(space.bns), max(space.ctas), 1)


def random_config(space: Space, rng: random.Random) -> Config:
    return (rng.choice(space.bns), rng.choice(space.ctas), rng.choice(space.orders))


def mutate(c: Config, space: Space, rng: random.Random) -> Config:
    """Move one field (of those with a choice) to an adjacent allowed value."""
    axes = [a for a, vals in enumerate((space.bns, space.ctas, space.orders)) if len(vals) > 1]
    if not axes:
        return c
    a = rng.choice(axes)
    vals = (space.bns, space.ctas, space.orders)[a]
    i = vals.index(c[a])
    j = i + rng.choice((-1, 1))
    j = min(max(j, 0), len(vals) - 1)
    if j == i:
        j = i - 1 if i > 0 else i + 1
    out = list(c)
    out[a] = vals[j]
    return tuple(out)


@dataclass
class Result:
    best: Config
    best_ms: float
    default: Config
    default_ms: float
    history: list = field(default_factory=list)  # (generation, config, ms, passed)


def evolve(evaluate, space: Space, generations: int = 4, population: int = 6, keep: int = 2,
           seed: int = 0) -> Result:
    """evaluate(config) -> (ms, passed).  Each configuration is measured once.
    A configuration that fails the gate never becomes a parent and never wins."""
    rng = random.Random(seed)
    seen: dict = {}
    history = []

    def score(c, gen):
        if c not in seen:
            seen[c] = evaluate(c)
            history.append((gen, c, seen[c][0], seen[c][1]))
        return seen[c]

    d = default_config(space)
    pop = [d] + [random_config(space, rng) for _ in range(population - 1)]
    for gen in range(generations):
        scored = []
        for c in dict.fromkeys(pop):  # distinct, in order
            ms, ok = score(c, gen)
            if ok:
                scored.append((ms, c))
        scored.sort()
        parents = [c for _, c in scored[:keep]] or [d]
        pop = parents + [mutate(rng.choice(parents), space, rng) for _ in range(population - len(parents))]
    passed = sorted((ms, c) for c, (ms, ok) in seen.items() if ok)
    if not passed:
        raise RuntimeError("no configuration passed the accuracy gate (not even the default)")
    best_ms, best = passed[0]
    return Result(best, best_ms, d, seen[d][0], history)


def status_passes(status: int, where: str = "") -> bool:
    """Whether a candidate's runs left the workspace's sticky error word
    clear.  A candidate whose launch hit a bounded-wait timeout stopped early,
    so its time would look short: it fails the gate.  Invalid group sizes are
    the caller's error, not the candidate's: they raise."""
    if status == binding.GMM_ERR_GROUP_SIZES:
        raise RuntimeError(f"{where}: {binding.STATUS_NAMES[status]}")
    return status == binding.GMM_OK


def tune_fp8_fwd(xq, xs, wq, ws, group_sizes, fuse: bool = False, quant: bool = False, generations: int = 4,
                 population: int = 6, keep: int = 2, seed: int = 0, reps: int = 5, atol: float | None = None,
                 rtol: float | None = None, stream=None) -> Result:
    """Search gmm_fp8_tile_config for this problem on the current device.

    The inputs are those of ``binding.fp8_fwd``. ``quant`` tunes the fused
    forward that also writes h's FP8 cast (``fp8_fwd_swiglu_quant``, the wi
    launch of the MoE layer); its gate compares h, the codes and the scales
    bit for bit. Each candidate runs ``reps`` times after one untimed run,
    and its time is the median. With atol/rtol left None, the gate for the
    plain forward is bit-exact against the default's output; given, it is
    torch.allclose with them."""
    fuse = fuse or quant
    dev = xq.device
    M, K = xq.shape
    G, Nw, _ = wq.shape
    N = Nw // 2 if fuse else Nw
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    space = space_for(N, fuse, sms)
    st = torch.cuda.current_stream(dev) if stream is None else stream
    work = binding.group_metadata(group_sizes, M, stream=st)

    def run(c, outs):
        if quant:
            binding.fp8_fwd_swiglu_quant(xq, xs, wq, ws, None, workspace=work, stream=st, config=c, out=outs)
        else:
            binding.fp8_fwd(xq, xs, wq, ws, None, fuse=fuse, out=outs[0], workspace=work, stream=st, config=c)

    def alloc():
        if quant:
            return (torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                    torch.empty((M, N), dtype=torch.uint8, device=dev),
                    torch.empty((N // 128, M), dtype=torch.float32, device=dev))
        return (torch.empty((M, N), dtype=torch.bfloat16, device=dev),)

    ref = alloc()
    run(None, ref)
    st.synchronize()  # the comparisons below run on torch's current stream
    status = work.status(st)
    if status != binding.GMM_OK:
        raise RuntimeError(f"default configuration: {binding.STATUS_NAMES.get(status, status)}")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def same_bits(a, b):
        return torch.equal(a.view(torch.uint8), b.view(torch.uint8))

    def device_ok(where):
        return status_passes(work.status(st), where)

    def evaluate(c):
        outs = alloc()
        run(c, outs)
        st.synchronize()
        ok = device_ok(f"config {c}")
        if quant or (atol is None and rtol is None):
            ok = ok and all(same_bits(a, b) for a, b in zip(outs, ref))
        else:
            ok = ok and torch.allclose(outs[0].float(), ref[0].float(), atol=atol or 0.0, rtol=rtol or 0.0)
        times = []
        for _ in range(reps):
            flush.zero_()
            torch.cuda.current_stream(dev).synchronize()  # the flush, before the timed launch
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            run(c, outs)
            e1.record(st)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        ok = device_ok(f"config {c}, timed runs") and ok
        times.sort()
        return times[len(times) // 2], bool(ok)

    return evolve(evaluate, space, generations, population, keep, seed)


def main(argv=None):
    """Tune the production MoE layer's two FP8 launches on this GPU and print
    every measured configuration: the fused wi (G=256, M=65536, K=2048, W with
    2 x 512 columns, writing h and its FP8 cast) and wo (K=512, N=2048 on the
    FP8 cast of h).
    Inputs are the seeded synthetic production workload (Zipf(1.1) top-8
    routing, X N(0,1) with 1% x50 outliers, W N(0, 1/K))."""
    import argparse
    import json
    import math

    import numpy as np

    from .workloads import routing_sizes

    ap = argparse.ArgumentParser(description=main.__doc__)
    ap.add_argument("--generations", type=int, default=4)
    ap.add_argument("--population", type=int, default=6)
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--seed", type=int, default=0)
    args = ap.parse_args(argv)
    dev = torch.device("cuda:0")
    G, M, K, N = 256, 65536, 2048, 512
    gen = torch.Generator(device=dev).manual_seed(1234)
    sizes = torch.from_numpy(routing_sizes("prod_fp8").astype(np.int32)).to(dev)
    x = torch.randn(M, K, device=dev, generator=gen)
    x = torch.where(torch.rand(M, K, device=dev, generator=gen) < 0.01, x * 50, x).to(torch.bfloat16)
    w_wi = (torch.randn(G, K, 2 * N, device=dev, generator=gen) / math.sqrt(K)).to(torch.bfloat16)
    w_wo = (torch.randn(G, N, K, device=dev, generator=gen) / math.sqrt(N)).to(torch.bfloat16)
    xq, xs = binding.quantize_lhs(x)
    wq_wi, ws_wi = binding.quantize_rhs(w_wi)
    wq_wo, ws_wo = binding.quantize_rhs(w_wo)
    _, hq, hs = binding.fp8_fwd_swiglu_quant(xq, xs, wq_wi, ws_wi, sizes, with_h=False)
    out = {}
    for name, a, quant in [("wi_fused_cast", (xq, xs, wq_wi, ws_wi), True), ("wo", (hq, hs, wq_wo, ws_wo), False)]:
        r = tune_fp8_fwd(*a, sizes, quant=quant, generations=args.generations, population=args.population,
                         reps=args.reps, seed=args.seed)
        out[name] = {"best": list(r.best), "best_us": round(r.best_ms * 1e3, 1), "default": list(r.default),
                     "default_us": round(r.default_ms * 1e3, 1),
                     "measured": [{"generation": g, "config": list(c), "us": round(ms * 1e3, 1), "passed": ok}
                                  for g, c, ms, ok in r.history]}
    print(json.dumps({"device": torch.cuda.get_device_name(dev), "config_fields": ["bn", "ctas", "unit_order"],
                      **out}, indent=1))


if __name__ == "__main__":
    main()

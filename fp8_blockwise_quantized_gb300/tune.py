"""Tile autotuner for the FP8 forward and for tgmm.

The search follows "GEMM Kernel 性能优化十问", Q8 and Q9.4.  Tile choices are
found by a search over candidates measured on the real shapes (Q4: the fwd,
bwd and tgmm phases each get their own tiling). A candidate may win only
after an accuracy check, which a caller can loosen but never switch off.

The spaces are the library's tile configurations:
- ``gmm_fp8_tile_config`` (``fp8_space``): ``bn`` the weight columns of a
  work unit (128, 256); ``ctas`` the persistent CTAs; ``unit_order`` (1
  row-tile major, 2 column-block major); ``cta_group`` (1 one CTA per 128-row
  tile, 2 CTA pairs on 256-row tiles); ``stages`` the slots of the operand
  ring; ``tmem_bufs`` the TMEM partial buffers the MMA rotates through.
- ``gmm_tgmm_tile_config`` (``tgmm_space``): ``stages`` the CTA-pair
  kernel's ring slots, ``claim_ahead`` the units its scheduler claims ahead of
  the producer, ``max_batch`` the most small units per claim.
Each field takes values from a list, and a rule (the same one the library
applies before any launch) says which combinations exist.

The search is evolutionary. The first population holds the default and random
valid members. Each generation keeps the fastest members that pass the gate
and fills up with mutants of them: a mutant moves one field to a neighbouring
value and, where the rule then forbids the combination, moves as few other
fields as it must (by the smallest steps) to reach a valid one.

The gate compares a candidate's outputs with those of the default
configuration, bit for bit: every configuration computes the same sums in
the same order. A caller may loosen the FP8 gate to an atol/rtol bound.
A candidate whose launch ran out a bounded wait fails the gate (its time is
no measurement).

Timing uses CUDA events on the launching stream, after one untimed run, with
L2 flushed between runs. Everything measured runs in the library's kernels;
this module only chooses arguments.
"""
from __future__ import annotations

import itertools
import random
from dataclasses import dataclass, field

import torch

from . import binding

Config = tuple


@dataclass(frozen=True)
class Space:
    """A tile-configuration space: field names, the values each field may take
    (in order, so that neighbours are adjacent), the default, and a rule
    (config -> bool) for the combinations that exist."""
    names: tuple
    values: tuple
    default: tuple
    rule: object = None

    def valid(self, c: Config) -> bool:
        return self.rule is None or bool(self.rule(c))

    def contains(self, c: Config) -> bool:
        return (len(c) == len(self.names) and all(v in vals for v, vals in zip(c, self.values))
                and self.valid(c))

    def members(self) -> list:
        return [c for c in itertools.product(*self.values) if self.valid(c)]


def _even(n: int) -> int:
    return max(2, n - n % 2)


def fp8_space(N: int, fuse: bool, sms: int) -> Space:
    """gmm_fp8_tile_config for an output of N columns (fused: the gate/up
    weight with 2N columns).  bn 256 needs N % 256 == 0 or the fused weight,
    which has 256-column units only; CTA pairs need 256-column units and an
    even CTA count; the ring slots and TMEM buffers are the compiled ones."""
    bns = (256,) if fuse else ((128, 256) if N % 256 == 0 else (128,))
    ctas = tuple(sorted({_even(sms * f // 8) for f in (4, 5, 6, 7, 8)}))
    groups = (1, 2) if (fuse or N % 256 == 0) else (1,)

    def rule(c):
        bn, n_ctas, _, cg, st, tb = c
        if cg == 2:
            return bn == 256 and n_ctas % 2 == 0 and 3 <= st <= (5 if fuse else 4) and tb == 4
        if bn == 256:
            return st in (2, 3) and tb == 2
        return st in (3, 4, 5) and tb in (2, 4)

    bn0 = max(bns)
    return Space(("bn", "ctas", "unit_order", "cta_group", "stages", "tmem_bufs"),
                 (bns, ctas, (1, 2), groups, (2, 3, 4, 5), (2, 4)),
                 (bn0, max(ctas), 1, 1, 3 if bn0 == 256 else 4, 2), rule)


def tgmm_space(K: int, N: int) -> Space:
    """gmm_tgmm_tile_config for dW [K, N]: the ring depth is selectable for
    the CTA-pair kernel with 256-column units (K % 256 == 0, N % 256 == 0)."""
    stages = (4, 5, 6) if (K % 256 == 0 and N % 256 == 0) else (6,)
    return Space(("stages", "claim_ahead", "max_batch"), (stages, (1, 2, 3, 4, 6, 8), (1, 2, 4)), (6, 3, 4))


def space_for(N: int, fuse: bool, sms: int) -> Space:
    return fp8_space(N, fuse, sms)


def default_config(space: Space) -> Config:
    return space.default


def random_config(space: Space, rng: random.Random) -> Config:
    return rng.choice(space.members())


def mutate(c: Config, space: Space, rng: random.Random) -> Config:
    """Move one field (of those with a choice) to an adjacent value; when the
    rule forbids the result, move the fewest other fields, by the smallest
    steps, to a valid combination.  Returns c itself only when no field can
    move."""
    moves = []
    for a, vals in enumerate(space.values):
        i = vals.index(c[a])
        for j in (i - 1, i + 1):
            if 0 <= j < len(vals):
                moves.append((a, vals[j]))
    rng.shuffle(moves)
    members = space.members()
    for a, v in moves:
        cands = [m for m in members if m[a] == v]
        if not cands:
            continue

        def cost(m, a=a):
            changed = [k for k in range(len(c)) if k != a and m[k] != c[k]]
            steps = sum(abs(space.values[k].index(m[k]) - space.values[k].index(c[k])) for k in changed)
            return (len(changed), steps)

        best = min(cost(m) for m in cands)
        return rng.choice([m for m in cands if cost(m) == best])
    return c


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


def _measure(space, work, st, dev, run, alloc, same, reps, generations, population, keep, seed) -> Result:
    """The search with the gate against the default configuration's outputs:
    run(config, outs) launches; alloc() -> fresh outputs; same(outs, ref)."""
    ref = alloc()
    run(None, ref)
    st.synchronize()
    status = work.status(st)
    if status != binding.GMM_OK:
        raise RuntimeError(f"default configuration: {binding.STATUS_NAMES.get(status, status)}")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def evaluate(c):
        outs = alloc()
        run(c, outs)
        st.synchronize()
        ok = status_passes(work.status(st), f"config {c}") and same(outs, ref)
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
        ok = status_passes(work.status(st), f"config {c}, timed runs") and ok
        times.sort()
        return times[len(times) // 2], bool(ok)

    return evolve(evaluate, space, generations, population, keep, seed)


def _same_bits(outs, ref):
    return all(torch.equal(a.view(torch.uint8), b.view(torch.uint8)) for a, b in zip(outs, ref))


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
    space = fp8_space(N, fuse, sms)
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

    def same(outs, ref):
        if quant or (atol is None and rtol is None):
            return _same_bits(outs, ref)
        return torch.allclose(outs[0].float(), ref[0].float(), atol=atol or 0.0, rtol=rtol or 0.0)

    return _measure(space, work, st, dev, run, alloc, same, reps, generations, population, keep, seed)


def tune_tgmm(x, dy, group_sizes, generations: int = 4, population: int = 6, keep: int = 2, seed: int = 0,
              reps: int = 5, stream=None) -> Result:
    """Search gmm_tgmm_tile_config for dW = X_g^T dY_g on the current device;
    the gate compares dW with the default configuration's bit for bit."""
    dev = x.device
    M, K = x.shape
    _, N = dy.shape
    G = group_sizes.numel()
    space = tgmm_space(K, N)
    st = torch.cuda.current_stream(dev) if stream is None else stream
    work = binding.group_metadata(group_sizes, M, stream=st)

    def run(c, outs):
        binding.tgmm(x, dy, None, dw=outs[0], workspace=work, stream=st, config=c)

    def alloc():
        return (torch.empty((G, K, N), dtype=torch.bfloat16, device=dev),)

    return _measure(space, work, st, dev, run, alloc, _same_bits, reps, generations, population, keep, seed)


def main(argv=None):
    """Tune the production MoE layer's launches on this GPU and print every
    measured configuration: the fused wi (G=256, M=65536, K=2048, W with
    2 x 512 columns, writing h and its FP8 cast), wo (K=512, N=2048 on the
    FP8 cast of h), and the two weight gradients (dW_wo = h^T dY with
    K=512, N=2048; dW_wi = X^T dH with K=2048, N=1024).
    Inputs are the seeded synthetic production workload (Zipf(1.1) top-8
    routing, X N(0,1) with 1% x50 outliers, W N(0, 1/K), dY and dH N(0,1))."""
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
    ap.add_argument("--only", default=None, help="comma-separated subset of wi_fused_cast,wo,tgmm_wo,tgmm_wi")
    args = ap.parse_args(argv)
    only = set(args.only.split(",")) if args.only else None
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
    del w_wi, w_wo
    h, hq, hs = binding.fp8_fwd_swiglu_quant(xq, xs, wq_wi, ws_wi, sizes)
    out = {}

    def record(name, r, fields):
        out[name] = {"fields": list(fields), "best": list(r.best), "best_us": round(r.best_ms * 1e3, 1),
                     "default": list(r.default), "default_us": round(r.default_ms * 1e3, 1),
                     "measured": [{"generation": g, "config": list(c), "us": round(ms * 1e3, 1), "passed": ok}
                                  for g, c, ms, ok in r.history]}

    kw = dict(generations=args.generations, population=args.population, reps=args.reps, seed=args.seed)
    fp8_fields = fp8_space(N, True, 2).names
    for name, a, quant in [("wi_fused_cast", (xq, xs, wq_wi, ws_wi), True), ("wo", (hq, hs, wq_wo, ws_wo), False)]:
        if only is None or name in only:
            record(name, tune_fp8_fwd(*a, sizes, quant=quant, **kw), fp8_fields)
    tgmm_fields = tgmm_space(256, 256).names
    if only is None or "tgmm_wo" in only:
        dy = torch.randn(M, K, device=dev, generator=gen).to(torch.bfloat16)
        record("tgmm_wo", tune_tgmm(h, dy, sizes, **kw), tgmm_fields)
        del dy
    if only is None or "tgmm_wi" in only:
        dh = torch.randn(M, 2 * N, device=dev, generator=gen).to(torch.bfloat16)
        record("tgmm_wi", tune_tgmm(x, dh, sizes, **kw), tgmm_fields)
    print(json.dumps({"device": torch.cuda.get_device_name(dev), **out}, indent=1))


if __name__ == "__main__":
    main()

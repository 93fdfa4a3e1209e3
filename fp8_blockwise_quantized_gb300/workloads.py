"""Seeded synthetic inputs for the MoE grouped matmul, shared by the tests, the
benchmark and the CPU oracle's callers.

This module holds no arithmetic of the method (no quantization, no GEMM, no
scale): only random numbers, their rounding to bf16 *as inputs*, and routing
counts.  Shapes follow the production-shape derivation of "GEMM Kernel
性能优化十问" Q6 (M = batch x seq x top_k; K = embedding dim; N = expert MLP
dim; G = experts; the development shape is one EP=8 shard of it).

Every array is produced on the host with numpy's PCG64 generator, so the same
seed gives the same bytes on any machine.  bf16 values are returned as
``numpy.uint16`` bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits.

    Inputs are finite by construction.
    """
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    hi = (u >> 16).astype(np.uint32)
    lo = u & 0xFFFF
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & 1) == 1))
    return (hi + up.astype(np.uint32)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------
# routing -> group_sizes
# ----------------------------------------------------------------------------

def routing_softmax_topk(tokens: int, experts: int, top_k: int, rng) -> np.ndarray:
    """Each token picks the top_k experts of softmax(N(0,1) logits).

    softmax is monotone, so the top_k of the logits is used directly; ties go
    to the lower expert id (stable sort).  Rows are then sorted by expert, so
    group g holds every (token, expert g) pair: group_sizes[g] = its count.
    """
    logits = rng.standard_normal((tokens, experts), dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    return np.bincount(order.ravel(), minlength=experts).astype(np.int32)


def routing_zipf(tokens: int, experts: int, top_k: int, alpha: float, n_dead: int,
                 rng) -> np.ndarray:
    """Zipf(alpha)-skewed expert popularity; top_k distinct experts per token.

    Popularity of the expert at rank r is r**-alpha; ranks are a random
    permutation of the experts.  The n_dead lowest-ranked experts get
    popularity 0, so their groups are empty.  Sampling without replacement
    in proportion to popularity uses the Gumbel-top-k construction.
    """
    ranks = rng.permutation(experts) + 1
    pop = ranks.astype(np.float64) ** (-alpha)
    if n_dead:
        pop[ranks > experts - n_dead] = 0.0
    with np.errstate(divide="ignore"):
        logp = np.log(pop / pop.sum())
    picks = np.empty((tokens, top_k), np.int64)
    chunk = 4096
    for t0 in range(0, tokens, chunk):
        t1 = min(tokens, t0 + chunk)
        gumbel = -np.log(-np.log(rng.random((t1 - t0, experts))))
        keys = logp[None, :] + gumbel
        picks[t0:t1] = np.argsort(-keys, axis=1, kind="stable")[:, :top_k]
    return np.bincount(picks.ravel(), minlength=experts).astype(np.int32)


def multinomial_sizes(M: int, G: int, empty: tuple[int, ...], rng) -> np.ndarray:
    p = np.ones(G)
    for g in empty:
        p[g] = 0.0
    return rng.multinomial(M, p / p.sum()).astype(np.int32)


# ----------------------------------------------------------------------------
# value generators
# ----------------------------------------------------------------------------

def normal_bf16(shape, std: float, rng, outlier_p: float = 0.0,
                outlier_scale: float = 50.0) -> np.ndarray:
    """bf16 N(0, std^2); each entry independently x outlier_scale with prob p."""
    v = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        v *= np.float32(std)
    if outlier_p > 0.0:
        mask = rng.random(shape, dtype=np.float32) < outlier_p
        v[mask] *= np.float32(outlier_scale)
    return f32_to_bf16_bits(v)


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------

@dataclass
class Case:
    name: str
    G: int
    M: int
    K: int
    N: int
    fuse: bool
    group_sizes: np.ndarray
    x: np.ndarray                      # bf16 bits [M, K]
    w: np.ndarray | None = None        # bf16 bits [G, K, N or 2N]
    dy: np.ndarray | None = None       # bf16 bits [M, N] (tgmm)
    w2: np.ndarray | None = None       # bf16 bits [G, N, K2] (second layer)
    N2: int = 0
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    "tiny_fp8": "G=4 M=512 K=256 N=256 fp8 fwd; group 2 empty",
    "wi_dev_fp8": "G=32 M=8192 K=2048 N=512 fp8 fwd; top-8 softmax routing, 1% x50 outliers",
    "wo_dev_fp8": "G=32 M=8192 K=512 N=2048 fp8 fwd; top-8 softmax routing, 1% x50 outliers",
    "tgmm_dev_bf16": "G=32 M=8192 K=2048 N=512 bf16 tgmm; top-8 softmax routing",
    "prod_fp8": ("G=256 M=65536 K=2048 N=2x512 fused silu*up, then K=512 N=2048; "
                 "Zipf(1.1) top-8 routing with 8 dead experts, 1% x50 outliers"),
}

SEED_BASE = 1000


def routing_sizes(name: str, seed: int | None = None) -> np.ndarray:
    idx = list(WORKLOADS).index(name)
    rng = np.random.default_rng(SEED_BASE + idx if seed is None else seed)
    if name == "tiny_fp8":
        return multinomial_sizes(512, 4, (2,), rng)
    if name in ("wi_dev_fp8", "wo_dev_fp8", "tgmm_dev_bf16"):
        return routing_softmax_topk(1024, 32, 8, rng)
    if name == "prod_fp8":
        return routing_zipf(8192, 256, 8, 1.1, 8, rng)
    raise KeyError(name)


def make_case(name: str, seed: int | None = None, with_second_layer: bool = True) -> Case:
    """Full-size inputs of one workload (host numpy arrays)."""
    idx = list(WORKLOADS).index(name)
    rng = np.random.default_rng(SEED_BASE + idx if seed is None else seed)
    if name == "tiny_fp8":
        G, M, K, N = 4, 512, 256, 256
        sizes = multinomial_sizes(M, G, (2,), rng)
        x = normal_bf16((M, K), 1.0, rng)
        w = normal_bf16((G, K, N), 1.0 / np.sqrt(K), rng)
        return Case(name, G, M, K, N, False, sizes, x, w)
    if name in ("wi_dev_fp8", "wo_dev_fp8"):
        G, M = 32, 8192
        K, N = (2048, 512) if name == "wi_dev_fp8" else (512, 2048)
        sizes = routing_softmax_topk(1024, G, 8, rng)
        x = normal_bf16((M, K), 1.0, rng, outlier_p=0.01)
        w = normal_bf16((G, K, N), 1.0 / np.sqrt(K), rng)
        return Case(name, G, M, K, N, False, sizes, x, w)
    if name == "tgmm_dev_bf16":
        G, M, K, N = 32, 8192, 2048, 512
        sizes = routing_softmax_topk(1024, G, 8, rng)
        x = normal_bf16((M, K), 1.0, rng)
        dy = normal_bf16((M, N), 1.0, rng)
        return Case(name, G, M, K, N, False, sizes, x, dy=dy)
    if name == "prod_fp8":
        G, M, K, N = 256, 65536, 2048, 512
        sizes = routing_zipf(8192, G, 8, 1.1, 8, rng)
        x = normal_bf16((M, K), 1.0, rng, outlier_p=0.01)
        w = normal_bf16((G, K, 2 * N), 1.0 / np.sqrt(K), rng)
        w2 = normal_bf16((G, N, K), 1.0 / np.sqrt(N), rng) if with_second_layer else None
        return Case(name, G, M, K, N, True, sizes, x, w, w2=w2, N2=K)
    raise KeyError(name)


def sample_rows(group_sizes: np.ndarray, per_group: int, rng) -> np.ndarray:
    """Sorted row indices: up to per_group rows of every non-empty group,
    always including each group's first and last row (ragged tile edges)."""
    off = np.concatenate([[0], np.cumsum(group_sizes.astype(np.int64))])
    rows = []
    for g in range(group_sizes.size):
        a, b = int(off[g]), int(off[g + 1])
        if b <= a:
            continue
        pick = {a, b - 1}
        if b - a > 2:
            extra = rng.choice(np.arange(a + 1, b - 1), size=min(per_group, b - a - 2),
                               replace=False)
            pick.update(int(r) for r in extra)
        rows.extend(sorted(pick))
    return np.array(rows, np.int64)


def subproblem_sizes(group_sizes: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """group_sizes of the GMM restricted to the sorted rows (rows stay grouped)."""
    off = np.concatenate([[0], np.cumsum(group_sizes.astype(np.int64))])
    g_of = np.searchsorted(off, rows, side="right") - 1
    return np.bincount(g_of, minlength=group_sizes.size).astype(np.int32)

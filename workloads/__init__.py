"""Seeded synthetic inputs for the proportional-PER workloads.

This module is the only thing the CUDA path (``cdf_scan_gb300``), its tests,
the bench and the CPU oracle share.  It draws random numbers and nothing
else: it holds none of the method's arithmetic (no powers, sums, searches or
weights).  Every generator is numpy's Philox bit generator seeded with the
workload's number, so any process on any machine draws the same inputs.

Workloads (sizes and distributions as stated for the method's benchmarks):

* ``small``     N=8192, p=|N(0,1)|+1e-6, alpha=0.6, beta=0.4, B=1024.
* ``minibatch`` N=262144, p=|N(0,1)|+1e-6, alpha=0.6; 32 rounds of
                build_cdf, sample 8192, update the 8192 sampled items with new
                |N(0,1)|+1e-6 priorities.
* ``tree``      capacity 500000 (2^19 leaves); initial fill 131072
                lognormal(0,1); 400 steps of insert 4096 lognormal(0,1) at the
                ring head, sample 1024, update 1024 with 20% duplicate indices.
* ``heavy``     N=1048576 lognormal(0, sigma=2) with 1% exact zeros,
                alpha=0.7, beta 0.4..1.0, B=65536.
* ``stress``    N=16777216 uniform(0,1], alpha=0.6, B=1048576; and
                ``resample``: 256 rows x 65536 log-weights N(0, sigma=2).
"""
from __future__ import annotations

import numpy as np


def rng(seed: int, stream: int = 0) -> np.random.Generator:
    """numpy Philox generator for workload ``seed``; ``stream`` picks an
    independent sub-stream (e.g. one per step of a loop)."""
    return np.random.Generator(np.random.Philox(key=[int(seed), int(stream)]))


def abs_normal(n: int, g: np.random.Generator, eps: float = 1e-6) -> np.ndarray:
    """|N(0,1)| + eps as float32."""
    return (np.abs(g.standard_normal(n)) + eps).astype(np.float32)


def lognormal(n: int, g: np.random.Generator, sigma: float = 1.0) -> np.ndarray:
    return g.lognormal(0.0, sigma, n).astype(np.float32)


def uniform_open_closed(n: int, g: np.random.Generator) -> np.ndarray:
    """uniform on (0,1]: 1 - U[0,1), drawn in float64 then rounded."""
    return (1.0 - g.random(n)).astype(np.float32)


# ---- the workloads ----------------------------------------------------------

SMALL = dict(name="small", N=8192, alpha=0.6, beta=0.4, B=1024, seed=1)
MINIBATCH = dict(name="minibatch", N=262144, alpha=0.6, beta=0.4, B=8192, rounds=32, seed=2)
TREE = dict(name="tree", capacity=500000, alpha=0.6, beta=0.4, initial=131072, insert=4096,
            B=1024, dup_frac=0.2, steps=400, seed=3)
HEAVY = dict(name="heavy", N=1048576, alpha=0.7, betas=(0.4, 0.5, 0.6, 0.7, 0.8, 0.9, 1.0),
             B=65536, zero_frac=0.01, sigma=2.0, seed=4)
STRESS = dict(name="stress", N=16777216, alpha=0.6, B=1048576, seed=5)
RESAMPLE = dict(name="resample", rows=256, P=65536, sigma=2.0, seed=6)


def small_priorities(N: int = SMALL["N"], seed: int = SMALL["seed"]) -> np.ndarray:
    return abs_normal(N, rng(seed))


def minibatch_priorities(N: int = MINIBATCH["N"], seed: int = MINIBATCH["seed"]) -> np.ndarray:
    return abs_normal(N, rng(seed))


def minibatch_new_priorities(round_: int, B: int = MINIBATCH["B"],
                             seed: int = MINIBATCH["seed"]) -> np.ndarray:
    """New |N(0,1)|+1e-6 priorities for the items sampled in round ``round_``."""
    return abs_normal(B, rng(seed, 1 + round_))


def tree_initial(n: int = TREE["initial"], seed: int = TREE["seed"]) -> np.ndarray:
    return lognormal(n, rng(seed))


def tree_insert(step: int, n: int = TREE["insert"], seed: int = TREE["seed"]) -> np.ndarray:
    return lognormal(n, rng(seed, 1 + 2 * step))


def tree_update_batch(step: int, sampled: np.ndarray, dup_frac: float = TREE["dup_frac"],
                      seed: int = TREE["seed"]):
    """Indices and new priorities for one update: the sampled indices with
    round(dup_frac*B) seeded positions overwritten by copies of other
    positions of the same batch (so those indices occur twice or more)."""
    g = rng(seed, 2 + 2 * step)
    idx = np.array(sampled, dtype=np.int32, copy=True)
    B = idx.size
    ndup = int(round(dup_frac * B))
    if B > 1 and ndup > 0:
        dst = g.choice(B, size=ndup, replace=False)
        src = g.integers(0, B, size=ndup)
        same = src == dst
        src[same] = (src[same] + 1) % B
        idx[dst] = idx[src]
    p = lognormal(B, g)
    return idx, p


def heavy_priorities(N: int = HEAVY["N"], seed: int = HEAVY["seed"],
                     sigma: float = HEAVY["sigma"], zero_frac: float = HEAVY["zero_frac"]) -> np.ndarray:
    g = rng(seed)
    p = lognormal(N, g, sigma)
    nz = int(round(zero_frac * N))
    p[g.choice(N, size=nz, replace=False)] = 0.0
    return p


def stress_priorities(N: int = STRESS["N"], seed: int = STRESS["seed"]) -> np.ndarray:
    return uniform_open_closed(N, rng(seed))


def resample_logw(rows: int = RESAMPLE["rows"], P: int = RESAMPLE["P"],
                  seed: int = RESAMPLE["seed"], sigma: float = RESAMPLE["sigma"]) -> np.ndarray:
    """rows x P log-weights N(0, sigma^2) as float32."""
    return (sigma * rng(seed).standard_normal((rows, P))).astype(np.float32)


def uniform01(n: int, seed: int, stream: int = 0) -> np.ndarray:
    """Explicit U[0,1) draws, for passing randomness in as an input."""
    return rng(seed, stream).random(n).astype(np.float32)

"""CPU checks of the seeded input recipes (the workload table of the design
notes): shapes, dtypes, seeding, and the distributions' stated parameters.
Small sizes keep the suite fast; the full-size generators are the same
functions with their default arguments."""
import math

import numpy as np
import pytest

import workloads


def test_the_same_seed_gives_the_same_inputs_and_streams_differ():
    a = workloads.small_priorities()
    b = workloads.small_priorities()
    assert np.array_equal(a, b)
    assert not np.array_equal(workloads.minibatch_new_priorities(0), workloads.minibatch_new_priorities(1))
    assert not np.array_equal(workloads.rng(7, 0).random(8), workloads.rng(7, 1).random(8))


def test_abs_normal_recipe():
    p = workloads.small_priorities()
    assert p.dtype == np.float32 and p.shape == (workloads.SMALL["N"],)
    assert np.all(p >= np.float32(1e-6))
    big = workloads.abs_normal(1 << 20, workloads.rng(11))
    assert abs(float(big.mean()) - (math.sqrt(2 / math.pi) + 1e-6)) < 3e-3  # E|N(0,1)|
    assert workloads.minibatch_priorities().shape == (workloads.MINIBATCH["N"],)
    assert workloads.minibatch_new_priorities(3).shape == (workloads.MINIBATCH["B"],)


def test_heavy_recipe_has_the_stated_zero_fraction_and_spread():
    n = 1 << 16
    p = workloads.heavy_priorities(N=n)
    assert p.dtype == np.float32
    assert int(np.sum(p == 0.0)) == round(workloads.HEAVY["zero_frac"] * n)
    logs = np.log(p[p > 0].astype(np.float64))
    assert abs(logs.std() - workloads.HEAVY["sigma"]) < 0.05  # lognormal(0, 2)
    assert abs(logs.mean()) < 0.05


def test_stress_recipe_is_uniform_on_open_closed_unit_interval():
    g = workloads.rng(workloads.STRESS["seed"])
    p = workloads.uniform_open_closed(1 << 20, g)
    assert p.dtype == np.float32
    assert float(p.min()) > 0.0 and float(p.max()) <= 1.0
    assert abs(float(p.mean()) - 0.5) < 2e-3
    # the full-size generator is the same recipe under the workload's seed
    assert np.array_equal(workloads.uniform_open_closed(1 << 10, workloads.rng(workloads.STRESS["seed"])),
                          workloads.stress_priorities(N=1 << 10))


def test_tree_update_batches_carry_the_stated_duplicates():
    B = workloads.TREE["B"]
    sampled = np.arange(B, dtype=np.int32) * 3
    idx, p = workloads.tree_update_batch(5, sampled)
    assert idx.dtype == np.int32 and p.dtype == np.float32 and idx.size == p.size == B
    ndup = round(workloads.TREE["dup_frac"] * B)
    # ndup positions were overwritten by copies of other positions
    assert B - np.unique(idx).size >= 1
    assert np.sum(idx != sampled) <= ndup
    assert set(idx.tolist()) <= set(sampled.tolist())
    assert workloads.tree_initial(n=1000).shape == (1000,)
    assert workloads.tree_insert(0, n=64).shape == (64,)


def test_resample_recipe():
    lw = workloads.resample_logw(rows=4, P=1 << 14)
    assert lw.dtype == np.float32 and lw.shape == (4, 1 << 14)
    assert abs(float(lw.std()) - workloads.RESAMPLE["sigma"]) < 0.05
    assert abs(float(lw.mean())) < 0.05


@pytest.mark.parametrize("n,seed,stream", [(16, 1, 0), (1000, 9, 3)])
def test_explicit_uniforms_lie_in_the_unit_interval(n, seed, stream):
    # float64 draws in [0, 1) rounded to float32 (the top 2^-25 rounds to 1)
    u = workloads.uniform01(n, seed, stream)
    assert u.dtype == np.float32 and u.shape == (n,)
    assert float(u.min()) >= 0.0 and float(u.max()) <= 1.0
    assert np.array_equal(u, workloads.uniform01(n, seed, stream))

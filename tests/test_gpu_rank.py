"""GPU parity of rank-based PER against the oracle.

Bars:
  * the order (radix sort): bit-exact against the oracle's stable sort by
    descending priority, ties by index, on tie-heavy inputs that span many
    sort tiles and a ragged tail;
  * the rank CDF: within 2e-6 * total of the oracle's fp64 prefix sum of
    q^alpha, monotone, bit-exact for alpha = 0 (the counts 1..n);
  * sampled items: bit-exact against the oracle's search of the GPU's rank
    CDF, mapped through the oracle's order;
  * IS weights: within 1e-6 relative of the oracle's weights of the drawn
    ranks, largest weight exactly 1; the standalone and fused weights agree
    bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

per = pytest.importorskip("cdf_scan_gb300")
RANK = per.PER_RANK


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def tied_priorities(n, seed):
    """|N(0,1)| rounded to 1/8: heavy ties; every 97th item 0 and every 89th -0."""
    g = workloads.rng(seed, n)
    p = (np.round(np.abs(g.standard_normal(n)) * 8.0) / 8.0).astype(np.float32)
    p[::97] = 0.0
    p[5::89] = -0.0
    return p


def rank_ctx(p, alpha, capacity=None):
    ctx = per.PerContext(capacity or max(1, p.size), alpha, RANK)
    per.per_set_priorities(ctx.handle, dev(p))
    per.per_rank_build(ctx.handle)
    return ctx


@pytest.mark.parametrize("n", [1, 2, 3, 31, 4095, 4096, 4097, 100_003, 1 << 20, (1 << 20) + 17])
def test_rank_order_and_cdf_match_oracle(n):
    p = tied_priorities(n, 301)
    alpha = 0.7
    ctx = rank_ctx(p, alpha)
    order = host(per.read_rank_order(ctx.handle))
    assert np.array_equal(order, oracle.rank_order(p))
    c = host(per.read_rank_cdf(ctx.handle)).astype(np.float64)
    C = oracle.cdf64(oracle.rank_priorities(n), alpha)
    assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]
    assert np.all(np.diff(c) >= 0)
    assert per.per_total_host(ctx.handle, RANK) == np.float32(c[-1])
    assert per.per_check(ctx.handle) == 0


@pytest.mark.parametrize("n", [262_145, 300_001, 600_000, 2_000_003])
def test_rank_order_back_to_back_builds(n):
    """Sizes just above the one-launch sort, where every launch of a pass can
    be resident at once: several builds queued without a host sync, the
    priorities switched between them, each order bit-exact."""
    pa = tied_priorities(n, 305)
    pb = workloads.lognormal(n, workloads.rng(306, n))
    want = {0: oracle.rank_order(pa), 1: oracle.rank_order(pb)}
    ctx = per.PerContext(n, 0.6, RANK)
    da, db = dev(pa), dev(pb)
    for k in range(4):
        per.per_set_priorities(ctx.handle, da if k % 2 == 0 else db)
        for _ in range(3):
            per.per_rank_build(ctx.handle)
        assert np.array_equal(host(per.read_rank_order(ctx.handle)), want[k % 2])
    assert per.per_check(ctx.handle) == 0


def test_rank_order_distinct_values_and_rebuild_after_updates():
    n = 70_001
    p = workloads.lognormal(n, workloads.rng(302))
    ctx = rank_ctx(p, 1.0)
    assert np.array_equal(host(per.read_rank_order(ctx.handle)), oracle.rank_order(p))
    # new priorities for a batch with repeated indices: the last write wins
    g = workloads.rng(303)
    idx = g.integers(0, n, 5000).astype(np.int32)
    newp = (g.random(5000) * 3.0).astype(np.float32)
    per.per_update(ctx.handle, dev(idx), dev(newp))
    per.per_rank_build(ctx.handle)
    p2 = oracle.apply_updates(p, idx, newp)
    assert np.array_equal(host(per.read_rank_order(ctx.handle)), oracle.rank_order(p2))
    assert per.per_check(ctx.handle) == 0


def test_rank_cdf_alpha_zero_counts_and_size_change():
    p = tied_priorities(50_000, 304)
    ctx = rank_ctx(p, 0.0)
    assert np.array_equal(host(per.read_rank_cdf(ctx.handle)), np.arange(1, 50_001, dtype=np.float32))
    # a smaller size: the order covers the first n items and the CDF is rebuilt
    per.per_set_size(ctx.handle, 12_345)
    out = torch.empty(16, dtype=torch.int32, device="cuda")
    with pytest.raises(per.PerError):  # the order is stale until per_rank_build
        per.per_sample(ctx.handle, 16, 1, 0, RANK, out)
    per.per_rank_build(ctx.handle)
    assert np.array_equal(host(per.read_rank_order(ctx.handle)), oracle.rank_order(p[:12_345]))
    assert np.array_equal(host(per.read_rank_cdf(ctx.handle)), np.arange(1, 12_346, dtype=np.float32))
    assert per.per_check(ctx.handle) == 0


@pytest.mark.parametrize("n,B", [(1, 7), (4097, 256), (65_536, 8192), (262_144, 8192), (1 << 20, 32_768)])
def test_rank_sampling_and_weights_match_oracle(n, B):
    p = tied_priorities(n, 305 + n % 7)
    alpha, beta = 0.7, 0.5
    ctx = rank_ctx(p, alpha)
    c = host(per.read_rank_cdf(ctx.handle))
    order = oracle.rank_order(p)
    ranks, _ = oracle.sample_cdf_f32(c, B, 11, 500)
    # plain sampling
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, 11, 500, RANK, out)
    assert np.array_equal(host(out), order[ranks])
    # fused sampling + weights (one launch up to 262,144 items, two above)
    idx = torch.empty(B, dtype=torch.int32, device="cuda")
    w = torch.empty(B, dtype=torch.float32, device="cuda")
    per.per_sample_weighted(ctx.handle, B, 11, 500, RANK, beta, idx, w)
    assert np.array_equal(host(idx), order[ranks])
    got = host(w)
    want = oracle.is_weights(oracle.rank_priorities(n), n, alpha, ranks, beta)
    assert got.max() == 1.0
    assert np.max(np.abs(got / want - 1.0)) <= 1e-6
    # standalone weights of the items look their ranks up: the same bits
    w2 = torch.empty(B, dtype=torch.float32, device="cuda")
    per.per_is_weights(ctx.handle, idx, beta, w2)
    assert np.array_equal(host(w2), got)
    assert per.per_check(ctx.handle) == 0


def test_rank_step_equals_update_build_sample():
    n, B = 131_072, 4096
    p = tied_priorities(n, 306)
    alpha, beta = 0.6, 0.4
    ctx = rank_ctx(p, alpha)
    g = workloads.rng(307)
    cur = p.copy()
    for step in range(3):
        upd = g.integers(0, n, B).astype(np.int32)
        newp = (np.round(g.random(B) * 16.0) / 8.0).astype(np.float32)
        idx = torch.empty(B, dtype=torch.int32, device="cuda")
        w = torch.empty(B, dtype=torch.float32, device="cuda")
        per.per_step(ctx.handle, dev(upd), dev(newp), B, 13, step * B, RANK, beta, idx, w)
        cur = oracle.apply_updates(cur, upd, newp)
        order = oracle.rank_order(cur)
        assert np.array_equal(host(per.read_rank_order(ctx.handle)), order)
        c = host(per.read_rank_cdf(ctx.handle))
        ranks, _ = oracle.sample_cdf_f32(c, B, 13, step * B)
        assert np.array_equal(host(idx), order[ranks])
        want = oracle.is_weights(oracle.rank_priorities(n), n, alpha, ranks, beta)
        assert np.max(np.abs(host(w) / want - 1.0)) <= 1e-6
    assert per.per_check(ctx.handle) == 0


def test_rank_negative_priority_is_reported_and_wrong_modes_refused():
    p = tied_priorities(10_000, 308)
    p[1234] = -1.0
    ctx = rank_ctx(p, 0.7)
    assert per.per_check(ctx.handle) == 8  # PER_ERR_VALUE
    with pytest.raises(per.PerError):
        per.per_build_cdf(ctx.handle)  # no proportional CDF in a rank context
    out = torch.empty(4, dtype=torch.int32, device="cuda")
    with pytest.raises(per.PerError):
        per.per_sample(ctx.handle, 4, 0, 0, per.PER_SCAN, out)
    with pytest.raises(per.PerError):
        per.PerContext(16, 0.7, RANK | per.PER_SCAN)
    with pytest.raises(per.PerError):
        per.PerContext((1 << 24) + 1, 0.7, RANK)

"""GPU tests of the totals and of the failure paths, through the C ABI.

* per_total / per_total_host in tree mode read tree[1] (foxhunt "GPU Segment
  Tree for PER Sampling", section "Integration": total_priority is tree[1]):
  equal, bit for bit, to the root of the oracle's pairwise rebuild of the
  GPU's leaves, after a bulk load and after updates.
* An update index outside [0, capacity) records PER_ERR_VALUE and writes
  nothing for that entry (the valid entries of the batch still apply).
* A lost message (per_debug_drop_tile: a carry word or a tile record that is
  never published) makes the waits for it run out: the call records
  PER_ERR_TIMEOUT, the kernels finish, and the next call on the same context
  is correct again against the oracle.  The waits are bounded (about 2 s); no
  GPU is faulted, trapped or hung.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

per = pytest.importorskip("cdf_scan_gb300")
SCAN, TREE = per.PER_SCAN, per.PER_TREE
ERR_TIMEOUT, ERR_VALUE = 4, 8


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def new_ctx(p, alpha, flags, capacity=None):
    ctx = per.PerContext(capacity or p.size, alpha, flags)
    per.per_set_priorities(ctx.handle, dev(p))
    return ctx


# --------------------------------------------------------------- totals -----

@pytest.mark.parametrize("cap", [1, 5000, 1 << 19])
def test_tree_total_is_the_root(cap):
    g = workloads.rng(400, cap)
    p = workloads.lognormal(cap, g)
    alpha = 0.6
    ctx = new_ctx(p, alpha, SCAN | TREE)
    out = torch.empty(1, dtype=torch.float32, device="cuda")
    for step in range(3):
        tree = host(per.read_tree(ctx.handle))
        leaves = tree[tree.size // 2:]
        root = oracle.tree_build(leaves)[1]
        per.per_total(ctx.handle, TREE, out)
        assert host(out)[0] == root == tree[1], f"step {step}"
        assert per.per_total_host(ctx.handle, TREE) == root
        # and the total is the sum of p^alpha (fp32 pairwise against fp64)
        pa = oracle.pow_alpha64(p, alpha)
        assert abs(float(root) / pa.sum() - 1.0) <= 1e-5
        # the scan path's total is cdf[n-1]
        per.per_build_cdf(ctx.handle)
        cdf = host(per.read_cdf(ctx.handle))
        per.per_total(ctx.handle, SCAN, out)
        assert host(out)[0] == cdf[cap - 1] == per.per_total_host(ctx.handle, SCAN)
        # updates with duplicates, then the totals again
        n = min(cap, 1024)
        idx = g.integers(0, cap, size=n).astype(np.int32)
        newp = workloads.lognormal(n, g)
        per.per_update(ctx.handle, dev(idx), dev(newp))
        p = oracle.apply_updates(p, idx, newp)
    assert per.per_check(ctx.handle) == 0


# ------------------------------------------------------ out-of-range index ---

@pytest.mark.parametrize("flags", [SCAN, TREE, SCAN | TREE])
def test_update_index_out_of_range_records_value_error(flags):
    cap = 10000
    g = workloads.rng(401)
    p = workloads.abs_normal(cap, g)
    ctx = new_ctx(p, 0.6, flags)
    tree0 = host(per.read_tree(ctx.handle)) if flags & TREE else None
    # a batch of nothing but bad indices changes nothing
    bad = np.array([cap, cap + 5, -1, 2**31 - 1], np.int32)
    per.per_update(ctx.handle, dev(bad), dev(np.full(bad.size, 7.0, np.float32)))
    assert per.per_check(ctx.handle) == ERR_VALUE
    assert per.per_check(ctx.handle) == 0  # read and cleared
    assert np.array_equal(host(per.read_priorities(ctx.handle, cap)), p)
    if flags & TREE:
        assert np.array_equal(host(per.read_tree(ctx.handle)), tree0)
    # in a mixed batch the valid entries apply, the bad ones are skipped
    idx = np.array([3, cap, 17, -4, 3], np.int32)
    newp = np.array([1.5, 9.0, 2.5, 9.0, 4.5], np.float32)
    per.per_update(ctx.handle, dev(idx), dev(newp))
    assert per.per_check(ctx.handle) == ERR_VALUE
    want = p.copy()
    want[17] = 2.5
    want[3] = 4.5  # the last occurrence wins
    assert np.array_equal(host(per.read_priorities(ctx.handle, cap)), want)
    if flags & TREE:
        tree = host(per.read_tree(ctx.handle))
        assert np.array_equal(tree[1:], oracle.tree_build(tree[tree.size // 2:])[1:])


# ------------------------------------------------------------ timeouts ------

def check_cdf(ctx, p, alpha):
    c = host(per.read_cdf(ctx.handle))[:p.size]
    C = oracle.cdf64(p, alpha)
    assert np.all(np.diff(c) >= 0)
    assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]
    return c


@pytest.mark.parametrize("n,drop", [(100_000, 5), (1_000_000, 40), (3 * (1 << 20) + 11, 3)],
                         ids=["one-wave-2048", "one-wave-4096", "streaming"])
def test_lost_scan_message_times_out_and_the_context_recovers(n, drop):
    """one-wave scans: tile `drop` never publishes its carry word; streaming
    scan: tile `drop` never publishes its record (sum or inclusive prefix)."""
    alpha = 0.6
    p = workloads.abs_normal(n, workloads.rng(402, n))
    ctx = new_ctx(p, alpha, SCAN)
    per.per_debug_drop_tile(ctx.handle, drop)
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == ERR_TIMEOUT
    # the injection was for one call: the next build is correct, twice
    for _ in range(2):
        per.per_build_cdf(ctx.handle)
        assert per.per_check(ctx.handle) == 0
        check_cdf(ctx, p, alpha)


def test_lost_message_in_the_fused_step_times_out_and_the_context_recovers():
    """per_step's one cooperative launch (update, scan, sample, weights): a
    tile's carry word is lost, the lookbacks waiting for it run out, the
    step's grid barriers still complete; the next steps match the oracle."""
    W = workloads.MINIBATCH
    N, B, alpha, beta, seed = W["N"], W["B"], W["alpha"], W["beta"], W["seed"]
    p = workloads.minibatch_priorities()
    ctx = new_ctx(p, alpha, SCAN)
    idx = torch.empty(B, dtype=torch.int32, device="cuda")
    w = torch.empty(B, dtype=torch.float32, device="cuda")
    per.per_debug_drop_tile(ctx.handle, 7)
    per.per_step(ctx.handle, None, None, B, seed, 0, SCAN, beta, idx, w)
    assert per.per_check(ctx.handle) == ERR_TIMEOUT
    prev = None
    for r in range(1, 4):
        newp = workloads.minibatch_new_priorities(r)
        upd = prev if prev is not None else np.arange(B, dtype=np.int32)
        per.per_step(ctx.handle, dev(upd), dev(newp), B, seed, r * B, SCAN, beta, idx, w)
        assert per.per_check(ctx.handle) == 0
        p = oracle.apply_updates(p, upd, newp)
        assert np.array_equal(host(per.read_priorities(ctx.handle, N)), p)
        c = check_cdf(ctx, p, alpha)
        got = host(idx)
        assert np.array_equal(got, oracle.sample_cdf_f32(c, B, seed, r * B)[0])
        ww = host(w)
        assert ww.max() == 1.0
        assert np.max(np.abs(ww / oracle.is_weights(p, N, alpha, got, beta) - 1.0)) <= 1e-6
        prev = got


def test_drop_of_a_tile_the_call_does_not_have_changes_nothing():
    p = workloads.abs_normal(5000, workloads.rng(403))
    ctx = new_ctx(p, 0.6, SCAN)
    per.per_debug_drop_tile(ctx.handle, 10**9)
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == 0
    check_cdf(ctx, p, 0.6)
    with pytest.raises(per.PerError):
        per.per_debug_drop_tile(ctx.handle, -2)


# --------------------------------------------------- exact-carry range ------
# Carries are 128-bit fixed point with 60 fractional bits: a unit sum (the
# fp32 sum of a one-wave tile, or of a 512-item slice of the streaming scan)
# must stay below 2^44, else PER_ERR_RANGE; unit sums below 2^-60 do not reach
# the carries, so such units are clamped to the carry before them.
ERR_RANGE = 7


@pytest.mark.parametrize("n", [4096, (1 << 21) + 5], ids=["one-wave", "streaming"])
def test_unit_sum_at_2_44_records_range_error(n):
    p = np.ones(n, np.float32)
    p[512:1024] = 2.0 ** 35  # one 512-item block: a unit sum of 2^44 in either kernel
    ctx = new_ctx(p, 1.0, SCAN)
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == ERR_RANGE
    assert per.per_check(ctx.handle) == 0  # read and cleared
    # just below the bound: no error, and the CDF within the usual tolerance
    p[512:1024] = np.float32(2.0 ** 35 * (1 - 2.0 ** -20))
    per.per_set_priorities(ctx.handle, dev(p))
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == 0
    check_cdf(ctx, p, 1.0)


@pytest.mark.parametrize("n", [5000, (1 << 21) + 5], ids=["one-wave", "streaming"])
def test_unit_sums_below_2_minus_60_vanish_from_the_carries(n):
    # 2^-75: a 2048-item tile or a 512-item slice sums to at most 2^-64
    tiny = np.float32(2.0 ** -75)
    # only tiny values: every unit sum is below 2^-60, so the CDF is 0
    ctx = new_ctx(np.full(n, tiny, np.float32), 1.0, SCAN)
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == 0
    c = host(per.read_cdf(ctx.handle))[:n]
    assert np.all(c == 0.0)
    assert per.per_total_host(ctx.handle, SCAN) == 0.0
    # one unit item first: the tiny tail stays at 1.0, which is also the fp32
    # rounding of the exact prefix sums (1 + k 2^-75)
    p = np.full(n, tiny, np.float32)
    p[0] = 1.0
    per.per_set_priorities(ctx.handle, dev(p))
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == 0
    c = host(per.read_cdf(ctx.handle))[:n]
    assert np.all(c == 1.0)
    assert np.array_equal(c, oracle.cdf64(p, 1.0).astype(np.float32))

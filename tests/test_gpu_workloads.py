"""GPU parity at the workloads' full sizes, in the launch configurations
bench.py times, against the CPU oracle on the same seeded inputs.

Bars as in test_gpu_parity.py: indices bit-exact when the oracle searches the
GPU's CDF or tree; CDF within 2e-6 * total (N <= 1M) or 1e-5 * total (16M),
monotone; priorities after updates bit-exact (last occurrence wins); tree
nodes bit-exact against the oracle's pairwise rebuild of the GPU leaves; IS
weights within 1e-6 relative of the fp64 formula.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

per = pytest.importorskip("cdf_scan_gb300")
SCAN, TREE = per.PER_SCAN, per.PER_TREE


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def new_ctx(p, alpha, flags, capacity=None):
    ctx = per.PerContext(capacity or p.size, alpha, flags)
    per.per_set_priorities(ctx.handle, dev(p))
    return ctx


def band_check(C, idx_gpu, idx_ref, u, band):
    """Indices may differ only where u lies within `band` of a CDF value
    between them (C: the oracle's fp64 CDF); returns the number of such
    differences."""
    bad = np.nonzero(idx_gpu != idx_ref)[0]
    for k in bad:
        lo, hi = sorted((int(idx_gpu[k]), int(idx_ref[k])))
        lo = max(lo - 1, 0)
        gap = np.min(np.abs(C[lo:hi + 1] - float(u[k])))
        assert gap <= band, f"sample {k}: gpu {idx_gpu[k]} oracle {idx_ref[k]} gap {gap} > {band}"
    return len(bad)


# ------------------------------------------------------------ scan update ---

@pytest.mark.parametrize("n_upd", [1, 7, 8192, 8193, 50000])
def test_scan_update_last_writer_wins(n_upd):
    """Scan-only contexts (one cooperative launch: last-writer election, grid
    barrier, apply); unsorted indices with duplicates."""
    N = 262144
    g = workloads.rng(200, n_upd)
    p0 = workloads.abs_normal(N, g)
    ctx = new_ctx(p0, 0.6, SCAN)
    idx = g.integers(0, N, size=n_upd).astype(np.int32)
    if n_upd > 4:
        dup = g.choice(n_upd, n_upd // 5, replace=False)
        idx[dup] = idx[g.integers(0, n_upd, size=dup.size)]
    newp = workloads.abs_normal(n_upd, g)
    for _ in range(2):  # the second call runs on the next epoch of the winner slots
        per.per_update(ctx.handle, dev(idx), dev(newp))
        want = oracle.apply_updates(p0, idx, newp)
        assert np.array_equal(host(per.read_priorities(ctx.handle, N)), want)
        p0 = want
        newp = workloads.abs_normal(n_upd, g)
    assert per.per_check(ctx.handle) == 0


# ------------------------------------------------------- minibatch loop -----

def test_minibatch_loop_matches_oracle(band_report):
    """The bench step itself: N=262144, 32 rounds of build_cdf, sample 8192
    with IS weights (beta 0.4, per_sample_weighted), update 8192 at the
    sampled indices."""
    W = workloads.MINIBATCH
    N, B, R, alpha, beta, seed = W["N"], W["B"], W["rounds"], W["alpha"], W["beta"], W["seed"]
    p = workloads.minibatch_priorities()
    ctx = new_ctx(p, alpha, SCAN)
    idx = torch.empty(B, dtype=torch.int32, device="cuda")
    w = torch.empty(B, dtype=torch.float32, device="cuda")
    n_band = 0
    for r in range(R):
        per.per_build_cdf(ctx.handle)
        per.per_sample_weighted(ctx.handle, B, seed, r * B, SCAN, beta, idx, w)
        newp = workloads.minibatch_new_priorities(r)
        per.per_update(ctx.handle, idx, dev(newp))
        c = host(per.read_cdf(ctx.handle))[:N]
        C = oracle.cdf64(p, alpha)
        assert np.all(np.diff(c) >= 0)
        assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]
        got = host(idx)
        want, _ = oracle.sample_cdf_f32(c, B, seed, r * B)
        assert np.array_equal(got, want), f"round {r}"
        own, u64 = oracle.sample_cdf_f64(C, B, seed, r * B)
        n_band += band_check(C, got, own, u64, 2e-6 * C[-1])
        ww = host(w)
        assert ww.max() == 1.0
        assert np.max(np.abs(ww / oracle.is_weights(p, N, alpha, got, beta) - 1.0)) <= 1e-6
        p = oracle.apply_updates(p, got, newp)
        assert np.array_equal(host(per.read_priorities(ctx.handle, N)), p), f"round {r}"
    band_report(f"minibatch workload (N={N}, {R} rounds x B={B}), scan", n_band, R * B, "2e-6 total")
    assert per.per_check(ctx.handle) == 0


# ------------------------------------------------------------- stress -------

@pytest.mark.parametrize("alpha", [0.6, 1.0])
def test_stress_scan_and_sample_full_size(alpha, band_report):
    """N = 16,777,216 uniform(0,1]; B = 1,048,576 stratified samples."""
    S = workloads.STRESS
    p = workloads.stress_priorities()
    ctx = new_ctx(p, alpha, SCAN)
    per.per_build_cdf(ctx.handle)
    c = host(per.read_cdf(ctx.handle))[:p.size]
    assert np.all(np.diff(c) >= 0)
    C = oracle.cdf64(p, alpha)
    assert np.max(np.abs(c - C)) <= 1e-5 * C[-1]
    out = torch.empty(S["B"], dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, S["B"], 1, 0, SCAN, out)
    got = host(out)
    want, _ = oracle.sample_cdf_f32(c, S["B"], 1, 0)
    assert np.array_equal(got, want)
    # against the oracle's own fp64 CDF: differences only within the 1e-5
    # band of the 16M CDF tolerance
    own, u64 = oracle.sample_cdf_f64(C, S["B"], 1, 0)
    n_band = band_check(C, got, own, u64, 1e-5 * C[-1])
    band_report(f"stress workload (N={p.size}, B={S['B']}, alpha={alpha}), scan", n_band, S["B"], "1e-5 total")
    assert per.per_check(ctx.handle) == 0


def test_stress_all_ones_is_exact():
    """cdf[i] = i + 1 is exact in fp32 up to 2^24 = the stress size."""
    n = workloads.STRESS["N"]
    ctx = new_ctx(np.ones(n, np.float32), 0.6, SCAN)
    per.per_build_cdf(ctx.handle)
    assert np.array_equal(host(per.read_cdf(ctx.handle))[:n], np.arange(1, n + 1, dtype=np.float32))


def test_resample_full_size(band_report):
    """256 rows x 65,536 log-weights N(0, 2^2)."""
    R = workloads.RESAMPLE
    lw = workloads.resample_logw()
    out = torch.empty((R["rows"], R["P"]), dtype=torch.int32, device="cuda")
    cdf = torch.empty((R["rows"], R["P"]), dtype=torch.float32, device="cuda")
    per.per_resample(dev(lw), 6, 0, out, out_cdf=cdf)
    got, c = host(out), host(cdf)
    n_band = n_checked = 0
    for b in range(0, R["rows"], 5):  # every fifth row against the fp64 oracle
        U = oracle.u01_closed_open(6, 0, b)
        assert np.array_equal(got[b], oracle.resample_row_on_cdf(c[b], U))
        own, C, u = oracle.resample_row(lw[b], U)
        assert np.max(np.abs(c[b] - C)) <= 2e-6
        n_band += band_check(C, got[b], own, u, 2e-6)
        n_checked += R["P"]
    band_report(f"resample workload ({R['rows']} x {R['P']}, every 5th row), row CDF", n_band, n_checked,
                "2e-6 (row total 1)")
    assert np.all(np.diff(got, axis=1) >= 0)


# ---------------------------------------------------------------- heavy -----

def test_heavy_workload_scan_and_tree_with_beta_ramp(band_report):
    """N = 1,048,576 lognormal(0, 2) with 1% zeros, alpha 0.7, B = 65,536,
    beta 0.4 .. 1.0; both sampling paths."""
    Hv = workloads.HEAVY
    p = workloads.heavy_priorities()
    N, B, alpha = p.size, Hv["B"], Hv["alpha"]
    ctx = new_ctx(p, alpha, SCAN | TREE)
    per.per_build_cdf(ctx.handle)
    c = host(per.read_cdf(ctx.handle))[:N]
    C = oracle.cdf64(p, alpha)
    assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]
    a = torch.empty(B, dtype=torch.int32, device="cuda")
    b = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, Hv["seed"], 0, SCAN, a)
    per.per_sample(ctx.handle, B, Hv["seed"], 0, TREE, b)
    ia, ib = host(a), host(b)
    assert np.array_equal(ia, oracle.sample_cdf_f32(c, B, Hv["seed"], 0)[0])
    tree = host(per.read_tree(ctx.handle))
    assert np.array_equal(ib, oracle.sample_tree(tree, B, Hv["seed"], 0)[0])
    assert np.all(p[ia] > 0) and np.all(p[ib] > 0)
    # both paths against the oracle's own fp64 CDF (scan thresholds from the
    # fp64 total; the tree's from its root)
    own, u64 = oracle.sample_cdf_f64(C, B, Hv["seed"], 0)
    band_report(f"heavy workload (N={N}, B={B}), scan", band_check(C, ia, own, u64, 2e-6 * C[-1]), B,
                "2e-6 total")
    _, ut = oracle.sample_tree(tree, B, Hv["seed"], 0)
    own_t = np.minimum(np.searchsorted(C, ut.astype(np.float64), side="left"), N - 1)
    band_report(f"heavy workload (N={N}, B={B}), tree", band_check(C, ib, own_t, ut, 2e-6 * C[-1]), B,
                "2e-6 total")
    w = torch.empty(B, dtype=torch.float32, device="cuda")
    for beta in Hv["betas"]:
        for flags_idx in (a, b):
            per.per_is_weights(ctx.handle, flags_idx, beta, w)
            got = host(w)
            want = oracle.is_weights(p, N, alpha, host(flags_idx), beta)
            assert got.max() == 1.0
            assert np.max(np.abs(got / want - 1.0)) <= 1e-6
    assert per.per_check(ctx.handle) == 0


# ----------------------------------------------------------------- tree -----

def test_tree_workload_steps(band_report):
    """Capacity 500,000 (2^19 leaves): initial fill 131,072 lognormal(0,1),
    then the workload's 400 steps of insert 4096 at the ring head, sample
    1024, update 1024 with 20% duplicate indices.  Every sampled index
    bit-exact against the oracle's descent of the GPU tree, and within the
    boundary band of a search of the oracle's fp64 CDF of its own leaves;
    the whole tree bit-exact against the oracle's pairwise rebuild of the
    oracle's own leaves at checkpoints."""
    T = workloads.TREE
    cap, B, alpha = T["capacity"], T["B"], T["alpha"]
    prio = np.zeros(cap, np.float32)
    init = workloads.tree_initial()
    prio[:init.size] = init
    ctx = per.PerContext(cap, alpha, TREE)
    per.per_set_priorities(ctx.handle, dev(prio))
    size, head = init.size, init.size % cap
    per.per_set_size(ctx.handle, size)
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    steps = T["steps"]  # 400: the ring fills after ~91 steps and wraps
    n_band = 0
    for s in range(steps):
        ins = workloads.tree_insert(s)
        ins_idx = ((head + np.arange(ins.size)) % cap).astype(np.int32)
        per.per_update(ctx.handle, dev(ins_idx), dev(ins))
        prio = oracle.apply_updates(prio, ins_idx, ins)
        head = (head + ins.size) % cap
        size = min(size + ins.size, cap)
        per.per_set_size(ctx.handle, size)
        per.per_sample(ctx.handle, B, T["seed"], s * B, TREE, out)
        got = host(out)
        tree = host(per.read_tree(ctx.handle))
        want, ut = oracle.sample_tree(tree, B, T["seed"], s * B)
        assert np.array_equal(got, want), f"step {s}"
        assert np.all(got < size)
        if s % 20 == 0:  # the fp64 search of the oracle's own leaves
            C = np.cumsum(oracle.pow_alpha64(prio, alpha))
            own = np.minimum(np.searchsorted(C, ut.astype(np.float64), side="left"), cap - 1)
            n_band += band_check(C, got, own, ut, 2e-6 * C[-1])
        uidx, up = workloads.tree_update_batch(s, got)
        per.per_update(ctx.handle, dev(uidx), dev(up))
        prio = oracle.apply_updates(prio, uidx, up)
        if s % 50 == 49 or s == steps - 1:
            tree = host(per.read_tree(ctx.handle))
            leaves = tree[tree.size // 2:]
            want_leaves = oracle.tree_leaves(prio, alpha, tree.size // 2)
            d = np.abs(leaves.view(np.int32).astype(np.int64) - want_leaves.view(np.int32).astype(np.int64))
            assert d.max() <= 4, f"step {s}: leaves differ from pow beyond 4 ulp"
            assert np.array_equal(tree[1:], oracle.tree_build(leaves)[1:]), f"step {s}"
    band_report(f"tree workload (2^19 leaves, every 20th of {steps} steps x B={B}), tree", n_band,
                (steps + 19) // 20 * B, "2e-6 total")
    assert per.per_check(ctx.handle) == 0


# ------------------------------------------------ fused sample + weights ----

@pytest.mark.parametrize("N,B,flags", [(262144, 8192, SCAN), (1000, 37, SCAN), (262144, 1, SCAN),
                                       (1 << 20, 65536, SCAN), (262144, 8192, SCAN | TREE)])
def test_sample_weighted_equals_the_two_calls(N, B, flags):
    """per_sample_weighted gives per_sample + per_is_weights bit for bit (one
    cooperative launch on the scan path when the coarse index fits, else the
    two launches)."""
    p = workloads.heavy_priorities(N=N)
    ctx = new_ctx(p, 0.7, flags)
    per.per_build_cdf(ctx.handle)
    i1 = torch.empty(B, dtype=torch.int32, device="cuda")
    w1 = torch.empty(B, dtype=torch.float32, device="cuda")
    i2 = torch.empty(B, dtype=torch.int32, device="cuda")
    w2 = torch.empty(B, dtype=torch.float32, device="cuda")
    for beta in (0.4, 1.0):
        per.per_sample(ctx.handle, B, 9, 77, SCAN, i1)
        per.per_is_weights(ctx.handle, i1, beta, w1)
        per.per_sample_weighted(ctx.handle, B, 9, 77, SCAN, beta, i2, w2)
        assert np.array_equal(host(i1), host(i2))
        assert np.array_equal(host(w1), host(w2))
        got = host(w2)
        assert got.max() == 1.0
        want = oracle.is_weights(p, N, 0.7, host(i2), beta)
        assert np.max(np.abs(got / want - 1.0)) <= 1e-6
    assert per.per_check(ctx.handle) == 0


# ------------------------------------------- grid barriers across grid sizes ---

def test_grid_barriers_across_varying_batch_sizes():
    """One context, batches whose grid sizes change from call to call: the
    grid-barrier word is shared by launches of different grid sizes and must
    come back ready after each (no timeout, results still exact)."""
    N = 262144
    g = workloads.rng(404, N)
    p = workloads.abs_normal(N, g)
    ctx = new_ctx(p, 0.6, SCAN)
    for n_upd in (8192, 1000, 8192, 300, 50000, 8193):
        idx = g.integers(0, N, size=n_upd).astype(np.int32)
        newp = workloads.abs_normal(n_upd, g)
        per.per_update(ctx.handle, dev(idx), dev(newp))
        p = oracle.apply_updates(p, idx, newp)
        assert per.per_check(ctx.handle) == 0, f"update n={n_upd}"
        assert np.array_equal(host(per.read_priorities(ctx.handle, N)), p)
    per.per_build_cdf(ctx.handle)
    c = host(per.read_cdf(ctx.handle))[:N]
    for B in (8192, 1000, 8192, 37, 65536, 8192):
        i1 = torch.empty(B, dtype=torch.int32, device="cuda")
        w1 = torch.empty(B, dtype=torch.float32, device="cuda")
        w2 = torch.empty(B, dtype=torch.float32, device="cuda")
        per.per_sample_weighted(ctx.handle, B, 5, B, SCAN, 0.4, i1, w1)
        assert per.per_check(ctx.handle) == 0, f"sample_weighted B={B}"
        per.per_is_weights(ctx.handle, i1, 0.4, w2)
        assert per.per_check(ctx.handle) == 0, f"is_weights B={B}"
        want, _ = oracle.sample_cdf_f32(c, B, 5, B)
        assert np.array_equal(host(i1), want)
        assert np.array_equal(host(w1), host(w2))
        assert np.max(np.abs(host(w2) / oracle.is_weights(p, N, 0.6, want, 0.4) - 1.0)) <= 1e-6


# ------------------------------------------------------------- fused step ---

@pytest.mark.parametrize("N,B,n_upd,flags", [(262144, 8192, 8192, SCAN), (262144, 8192, 0, SCAN),
                                             (262144, 1, 5, SCAN), (1000, 37, 300, SCAN), (8192, 1024, 1024, SCAN),
                                             (262144, 65536, 8192, SCAN), (1 << 20, 8192, 4096, SCAN),
                                             (262144, 8192, 8192, SCAN | TREE)])
def test_per_step_equals_the_separate_calls(N, B, n_upd, flags):
    """per_step (one cooperative launch when it applies, else the separate
    calls) gives per_update + per_build_cdf + per_sample_weighted bit for
    bit: indices, weights, priorities and CDF, over several rounds."""
    g = workloads.rng(505, N + B + n_upd)
    p = workloads.abs_normal(N, g)
    a, b = new_ctx(p, 0.6, flags), new_ctx(p, 0.6, flags)
    ia = torch.empty(B, dtype=torch.int32, device="cuda")
    wa = torch.empty(B, dtype=torch.float32, device="cuda")
    ib = torch.empty(B, dtype=torch.int32, device="cuda")
    wb = torch.empty(B, dtype=torch.float32, device="cuda")
    for r in range(3):
        if n_upd:
            idx = g.integers(0, N, size=n_upd).astype(np.int32)
            if n_upd > 4:
                dup = g.choice(n_upd, n_upd // 5, replace=False)
                idx[dup] = idx[g.integers(0, n_upd, size=dup.size)]
            ui, up = dev(idx), dev(workloads.abs_normal(n_upd, g))
        else:
            ui = up = None
        u01 = dev(workloads.uniform_open_closed(B, g)) if r == 2 else None
        per.per_step(a.handle, ui, up, B, 11, r * B, SCAN, 0.4, ia, wa, u01=u01)
        if n_upd:
            per.per_update(b.handle, ui, up)
        per.per_build_cdf(b.handle)
        per.per_sample_weighted(b.handle, B, 11, r * B, SCAN, 0.4, ib, wb, u01=u01)
        assert np.array_equal(host(ia), host(ib)), f"round {r}"
        assert np.array_equal(host(wa), host(wb)), f"round {r}"
        assert np.array_equal(host(per.read_priorities(a.handle, N)), host(per.read_priorities(b.handle, N)))
        assert np.array_equal(host(per.read_cdf(a.handle))[:N], host(per.read_cdf(b.handle))[:N])
    assert per.per_check(a.handle) == 0
    assert per.per_check(b.handle) == 0


def test_per_step_heavy_duplicates_across_rounds():
    """20,000 updates (several rounds of the fused update) that all hit 300
    items around a tile boundary: the last occurrence of each index wins, as
    in per_update and in the oracle."""
    N, B, n_upd = 262144, 4096, 20000
    g = workloads.rng(506, 1)
    p = workloads.abs_normal(N, g)
    a, b = new_ctx(p, 0.6, SCAN), new_ctx(p, 0.6, SCAN)
    idx = (2048 * 37 - 150 + g.integers(0, 300, size=n_upd)).astype(np.int32)
    newp = workloads.abs_normal(n_upd, g)
    ia = torch.empty(B, dtype=torch.int32, device="cuda")
    wa = torch.empty(B, dtype=torch.float32, device="cuda")
    ib = torch.empty(B, dtype=torch.int32, device="cuda")
    wb = torch.empty(B, dtype=torch.float32, device="cuda")
    per.per_step(a.handle, dev(idx), dev(newp), B, 3, 0, SCAN, 0.4, ia, wa)
    per.per_update(b.handle, dev(idx), dev(newp))
    per.per_build_cdf(b.handle)
    per.per_sample_weighted(b.handle, B, 3, 0, SCAN, 0.4, ib, wb)
    want = oracle.apply_updates(p, idx, newp)
    assert np.array_equal(host(per.read_priorities(a.handle, N)), want)
    assert np.array_equal(host(per.read_priorities(b.handle, N)), want)
    assert np.array_equal(host(ia), host(ib))
    assert np.array_equal(host(wa), host(wb))
    assert per.per_check(a.handle) == 0


def test_minibatch_loop_with_per_step_matches_oracle():
    """The minibatch workload through per_step: round r applies round r-1's
    updates, rebuilds and samples; checked against the oracle every round."""
    W = workloads.MINIBATCH
    N, B, R, alpha, beta, seed = W["N"], W["B"], W["rounds"], W["alpha"], W["beta"], W["seed"]
    p = workloads.minibatch_priorities()
    ctx = new_ctx(p, alpha, SCAN)
    idx = [torch.empty(B, dtype=torch.int32, device="cuda") for _ in range(2)]
    w = torch.empty(B, dtype=torch.float32, device="cuda")
    newp = None
    for r in range(R):
        prev = idx[(r + 1) % 2] if r else None
        per.per_step(ctx.handle, prev, newp, B, seed, r * B, SCAN, beta, idx[r % 2], w)
        if r:
            p = oracle.apply_updates(p, host(prev), host(newp))
        c = host(per.read_cdf(ctx.handle))[:N]
        C = oracle.cdf64(p, alpha)
        assert np.all(np.diff(c) >= 0)
        assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]
        got = host(idx[r % 2])
        want, _ = oracle.sample_cdf_f32(c, B, seed, r * B)
        assert np.array_equal(got, want), f"round {r}"
        ww = host(w)
        assert ww.max() == 1.0
        assert np.max(np.abs(ww / oracle.is_weights(p, N, alpha, got, beta) - 1.0)) <= 1e-6
        newp = dev(workloads.minibatch_new_priorities(r))
    assert per.per_check(ctx.handle) == 0

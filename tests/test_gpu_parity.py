"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars (written in each test):
  * CDF: |cdf_gpu - C_oracle| <= 2e-6 * total for N <= 1M (1e-5 at 16M);
    monotone; bit-exact for all-ones and for integer priorities (alpha=1,
    total < 2^24); bit-identical across reruns.
  * scan-path indices: bit-exact when the oracle searches the GPU's CDF;
    against the oracle's own fp64 CDF, differences only where the threshold
    is within 2e-6*total of a boundary (count reported).
  * tree: every node bit-exact against the oracle's full pairwise rebuild of
    the GPU's leaves; leaves within 4 ulp of fl32(pow64); sampled indices
    bit-exact against the oracle's descent on the GPU tree.
  * IS weights within 1e-6 relative of the fp64 oracle; max weight exactly 1.
  * resampling: bit-exact on the GPU's row CDF; band rule against fp64.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

per = pytest.importorskip("cdf_scan_gb300")
SCAN, TREE = per.PER_SCAN, per.PER_TREE


def dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def make_ctx(p, alpha, flags=SCAN | TREE, capacity=None):
    ctx = per.PerContext(capacity or max(1, p.size), alpha, flags)
    per.per_set_priorities(ctx.handle, dev(p))
    return ctx


def gpu_cdf(p, alpha):
    ctx = make_ctx(p, alpha, SCAN)
    per.per_build_cdf(ctx.handle)
    c = host(per.read_cdf(ctx.handle))
    assert per.per_check(ctx.handle) == 0
    return ctx, c


def band_check(C, idx_gpu, idx_ref, u, band):
    """Indices may differ only where u lies within `band` of a CDF value
    between them; returns the number of such differences."""
    bad = np.nonzero(idx_gpu != idx_ref)[0]
    for k in bad:
        lo, hi = sorted((int(idx_gpu[k]), int(idx_ref[k])))
        lo = max(lo - 1, 0)
        gap = np.min(np.abs(C[lo:hi + 1] - float(u[k])))
        assert gap <= band, f"sample {k}: gpu {idx_gpu[k]} oracle {idx_ref[k]} gap {gap} > {band}"
    return len(bad)


# ------------------------------------------------------------------ CDF -----

@pytest.mark.parametrize("n", [1, 2, 3, 31, 32, 33, 127, 1023, 1024, 1025, 4095, 4096, 4097, 8192,
                               65537, 262144, 1048575, 1048577])
def test_cdf_matches_oracle_ragged_sizes(n):
    p = workloads.abs_normal(n, workloads.rng(100, n))
    alpha = 0.6
    _, c = gpu_cdf(p, alpha)
    C = oracle.cdf64(p, alpha)
    assert c.shape == (n,)
    assert np.all(np.diff(c) >= 0), "CDF must be non-decreasing"
    assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]


# Inputs beyond one wave of tiles take the streaming kernel (16384-item tiles
# by ticket, one CTA per SM): fewer tiles than CTAs, a last tile that ends
# exactly at n (item n-1 in a full tile), last tiles of 1 item (no bulk copy)
# and of 7 items (4 copied, 3 read directly), and several tiles per CTA.
STREAM_SIZES = [1_400_000, 1 << 21, (1 << 21) + 1, (1 << 21) + 7, 5_000_000, 4 * 152 * 16384 + 5]


@pytest.mark.parametrize("n", STREAM_SIZES)
def test_cdf_streaming_path_ragged(n):
    p = workloads.abs_normal(n, workloads.rng(104, n))
    ctx, c = gpu_cdf(p, 0.6)
    C = oracle.cdf64(p, 0.6)
    assert np.all(np.diff(c) >= 0)
    assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]
    assert per.per_total_host(ctx.handle, SCAN) == c[-1]


@pytest.mark.parametrize("alpha", [0.0, 1.0])
def test_cdf_streaming_path_exact_modes(alpha):
    # alpha = 0 counts items (0^0 = 1); alpha = 1 on small integers is exact
    n = (1 << 21) + 3
    p = workloads.rng(105).integers(0, 5, size=n).astype(np.float32)  # total < 2^24
    _, c = gpu_cdf(p, alpha)
    want = np.arange(1, n + 1) if alpha == 0.0 else np.cumsum(p.astype(np.int64))
    assert np.array_equal(c, want.astype(np.float32))


def test_cdf_streaming_path_reports_negative_priority():
    # alpha = 1: the slice sums stay finite, so only PER_ERR_VALUE is recorded
    # (with a fractional alpha the power of -1 is NaN and the range check
    # fires first)
    p = np.ones((1 << 21) + 5, np.float32)
    p[1_234_567] = -1.0
    ctx = make_ctx(p, 1.0, SCAN)
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == 8  # PER_ERR_VALUE
    per.per_set_priorities(ctx.handle, dev(np.abs(p)))
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == 0


def test_cdf_streaming_path_repeated_calls_and_sizes():
    # repeated streaming scans on one context, the size changing between
    # calls: records of earlier calls (more tiles, other sums) carry older
    # tags and are never taken; every call equals the first one of its size
    cap = (1 << 22) + 9
    p = workloads.abs_normal(cap, workloads.rng(106))
    ctx = make_ctx(p, 0.6, SCAN)
    first = {}
    for rep in range(3):
        for size in (cap, 3 * (1 << 20) + 5, (1 << 21) + 1, cap):
            per.per_set_size(ctx.handle, size)
            per.per_build_cdf(ctx.handle)
            assert per.per_check(ctx.handle) == 0
            c = host(per.read_cdf(ctx.handle))[:size]
            if size not in first:
                C = oracle.cdf64(p[:size], 0.6)
                assert np.all(np.diff(c) >= 0)
                assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]
                first[size] = c
            else:
                assert np.array_equal(c, first[size]), (rep, size)


def test_cdf_large_tile_path_ragged():
    # lognormal priorities through the streaming kernel; ragged tail included
    n = 3 * 1024 * 1024 + 12345
    p = workloads.lognormal(n, workloads.rng(101), 1.0)
    _, c = gpu_cdf(p, 0.7)
    C = oracle.cdf64(p, 0.7)
    assert np.all(np.diff(c) >= 0)
    assert np.max(np.abs(c - C)) <= 2e-6 * C[-1]


@pytest.mark.parametrize("n", [1, 4096, 1 << 20, (1 << 22) + 3])
def test_cdf_all_ones_exact(n):
    _, c = gpu_cdf(np.ones(n, np.float32), 0.6)
    assert np.array_equal(c, np.arange(1, n + 1, dtype=np.float32))


def test_cdf_integer_priorities_alpha_one_exact():
    g = workloads.rng(102)
    p = g.integers(0, 8, size=1_000_003).astype(np.float32)  # total < 2^24
    _, c = gpu_cdf(p, 1.0)
    assert np.array_equal(c, np.cumsum(p.astype(np.int64)).astype(np.float32))


def test_cdf_zero_alpha_counts_items():
    p = workloads.heavy_priorities(N=50_000)  # zeros included: 0^0 = 1
    _, c = gpu_cdf(p, 0.0)
    assert np.array_equal(c, np.arange(1, p.size + 1, dtype=np.float32))


def test_cdf_bit_reproducible():
    p = workloads.heavy_priorities(N=1 << 20)
    ctx = make_ctx(p, 0.7, SCAN)
    per.per_build_cdf(ctx.handle)
    first = host(per.read_cdf(ctx.handle))
    for _ in range(20):
        per.per_build_cdf(ctx.handle)
        assert np.array_equal(host(per.read_cdf(ctx.handle)), first)
    assert per.per_check(ctx.handle) == 0


def test_cdf_total_matches_per_total():
    p = workloads.small_priorities()
    ctx, c = gpu_cdf(p, 0.6)
    assert per.per_total_host(ctx.handle, SCAN) == c[-1]
    out = torch.zeros(1, device="cuda")
    per.per_total(ctx.handle, SCAN, out)
    assert host(out)[0] == c[-1]


# ----------------------------------------------------------- scan sampler ---

@pytest.mark.parametrize("N,B", [(8192, 1024), (262144, 8192), (1000, 1), (1000, 777), (5000, 20000),
                                 (1 << 20, 65536), (33, 1024)])
def test_sample_scan_bit_exact_on_gpu_cdf(N, B, band_report):
    p = workloads.abs_normal(N, workloads.rng(103, N))
    ctx, c = gpu_cdf(p, 0.6)
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, seed=7, offset=1000, mode=SCAN, out_idx=out)
    got = host(out)
    want, u = oracle.sample_cdf_f32(c, B, 7, 1000)
    assert np.array_equal(got, want)
    assert np.all(np.diff(got) >= 0)
    # against the oracle's own fp64 CDF: only boundary-band differences
    C = oracle.cdf64(p, 0.6)
    own, u64 = oracle.sample_cdf_f64(C, B, 7, 1000)
    n_band = band_check(C, got, own, u64, 2e-6 * C[-1])
    name = "small workload (N=8192, B=1024), scan" if (N, B) == (8192, 1024) else f"scan N={N} B={B}"
    band_report(name, n_band, B, "2e-6 total")
    # an fp32 CDF cannot resolve boundaries closer than ~1 ulp of the total:
    # expect about (N * 1e-7) of the samples to sit that close to one
    assert n_band <= B * (1e-7 * N + 1e-3) + 2
    assert per.per_check(ctx.handle) == 0


def test_sample_scan_u01_override_and_zero_priorities():
    p = workloads.heavy_priorities(N=100_000)
    ctx, c = gpu_cdf(p, 0.7)
    B = 4096
    u01 = (1.0 - workloads.uniform01(B, 104)).astype(np.float32)  # (0, 1]
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, 0, 0, SCAN, out, u01=dev(u01))
    got = host(out)
    want, _ = oracle.sample_cdf_f32(c, B, 0, 0, u01=u01)
    assert np.array_equal(got, want)
    assert np.all(p[got] > 0), "a zero-priority item was drawn"


# ------------------------------------------------------------------ tree ----

def ulp_diff(a, b):
    a = np.asarray(a, np.float32).view(np.int32).astype(np.int64)
    b = np.asarray(b, np.float32).view(np.int32).astype(np.int64)
    return np.abs(a - b)


def check_tree(ctx, raw_prio, alpha):
    tree = host(per.read_tree(ctx.handle))
    cap = tree.size // 2
    leaves = tree[cap:]
    want_leaves = oracle.tree_leaves(raw_prio, alpha, cap)
    assert np.max(ulp_diff(leaves, want_leaves)) <= 4
    rebuilt = oracle.tree_build(leaves)
    assert np.array_equal(tree[1:], rebuilt[1:]), "internal sums differ from the pairwise rebuild"
    return tree


@pytest.mark.parametrize("cap", [1, 2, 5, 4096, 500000])
def test_tree_build_from_priorities(cap):
    p = workloads.lognormal(cap, workloads.rng(105, cap))
    ctx = make_ctx(p, 0.6, TREE)
    check_tree(ctx, p, 0.6)
    assert per.per_check(ctx.handle) == 0


@pytest.mark.parametrize("n_upd", [1, 17, 1024, 1025, 4096])
def test_tree_update_last_writer_wins(n_upd):
    cap = 500000
    g = workloads.rng(106, n_upd)
    p0 = workloads.lognormal(cap, g)
    ctx = make_ctx(p0, 0.6, TREE | SCAN)
    idx = g.integers(0, cap, size=n_upd).astype(np.int32)
    if n_upd > 4:
        dup = g.choice(n_upd, n_upd // 5, replace=False)
        idx[dup] = idx[g.integers(0, n_upd, size=dup.size)]
    newp = workloads.lognormal(n_upd, g)
    per.per_update(ctx.handle, dev(idx), dev(newp))
    want_raw = oracle.apply_updates(p0, idx, newp)
    got_raw = host(per.read_priorities(ctx.handle, cap))
    assert np.array_equal(got_raw, want_raw)
    check_tree(ctx, want_raw, 0.6)
    assert per.per_check(ctx.handle) == 0


def test_tree_update_is_deterministic_across_reruns():
    cap = 1 << 19
    p0 = workloads.lognormal(cap, workloads.rng(107))
    g = workloads.rng(108)
    idx = g.integers(0, cap, size=1024).astype(np.int32)
    idx[:200] = idx[200:400]
    newp = workloads.lognormal(1024, g)
    trees = []
    for _ in range(5):
        ctx = make_ctx(p0, 0.6, TREE)
        per.per_update(ctx.handle, dev(idx), dev(newp))
        trees.append(host(per.read_tree(ctx.handle)))
    for t in trees[1:]:
        assert np.array_equal(t, trees[0])


@pytest.mark.parametrize("cap,B", [(8192, 1024), (500000, 1024), (1 << 20, 65536), (3, 100)])
def test_tree_sample_bit_exact(cap, B):
    p = workloads.heavy_priorities(N=cap) if cap > 10 else np.array([1.0, 0.0, 2.0], np.float32)
    ctx = make_ctx(p, 0.7, TREE)
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, 11, 5, TREE, out)
    got = host(out)
    tree = host(per.read_tree(ctx.handle))
    want, _ = oracle.sample_tree(tree, B, 11, 5)
    assert np.array_equal(got, want)
    assert np.all(p[got] > 0)


def test_tree_and_scan_agree_except_in_band():
    p = workloads.heavy_priorities()  # 1M, lognormal(0,2), 1% zeros
    B = 65536
    ctx = make_ctx(p, 0.7, SCAN | TREE)
    per.per_build_cdf(ctx.handle)
    a = torch.empty(B, dtype=torch.int32, device="cuda")
    b = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, 3, 0, SCAN, a)
    per.per_sample(ctx.handle, B, 3, 0, TREE, b)
    ia, ib = host(a), host(b)
    C = oracle.cdf64(p, 0.7)
    _, u = oracle.sample_cdf_f64(C, B, 3, 0)
    n = band_check(C, ia, ib, u, 4e-6 * C[-1])
    assert n <= B * (2e-7 * p.size + 1e-3)


# ------------------------------------------------------------ IS weights ----

@pytest.mark.parametrize("flags", [SCAN, TREE])
@pytest.mark.parametrize("B", [1, 1024, 8192, 8193, 65536, 1 << 20])
def test_is_weights_match_fp64(flags, B):
    N = max(B, 8192)
    p = workloads.heavy_priorities(N=N)
    ctx = make_ctx(p, 0.7, flags)
    if flags == SCAN:
        per.per_build_cdf(ctx.handle)
    idx = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, 21, 0, flags, idx)
    for beta in (0.4, 1.0):
        w = torch.empty(B, dtype=torch.float32, device="cuda")
        per.per_is_weights(ctx.handle, idx, beta, w)
        got = host(w)
        want = oracle.is_weights(p, N, 0.7, host(idx), beta)
        assert got.max() == 1.0
        assert np.max(np.abs(got / want - 1.0)) <= 1e-6
    assert per.per_check(ctx.handle) == 0


def test_is_weights_equal_priorities_and_beta_zero():
    p = np.full(4096, 2.5, np.float32)
    ctx = make_ctx(p, 0.6, TREE)
    idx = dev(np.arange(0, 4096, 3, dtype=np.int32))
    w = torch.empty(idx.numel(), device="cuda")
    per.per_is_weights(ctx.handle, idx, 0.7, w)
    assert np.all(host(w) == 1.0)
    p2 = workloads.lognormal(4096, workloads.rng(109))
    ctx2 = make_ctx(p2, 0.6, TREE)
    per.per_is_weights(ctx2.handle, idx, 0.0, w)
    assert np.all(host(w) == 1.0)


# -------------------------------------------------------------- resample ----

@pytest.mark.parametrize("rows,P", [(1, 4), (3, 1024), (4, 4100), (16, 65536), (5, 5 * 4096 + 100),
                                    (2, 3 * 4096 + 4)])
def test_resample_matches_oracle(rows, P):
    lw = workloads.resample_logw(rows=rows, P=P, seed=110 + rows)
    out = torch.empty((rows, P), dtype=torch.int32, device="cuda")
    cdf = torch.empty((rows, P), dtype=torch.float32, device="cuda")
    per.per_resample(dev(lw), 9, 100, out, out_cdf=cdf)
    got, c = host(out), host(cdf)
    for b in range(rows):
        U = oracle.u01_closed_open(9, 100, b)
        assert np.array_equal(got[b], oracle.resample_row_on_cdf(c[b], U))
        want, C, u = oracle.resample_row(lw[b], U)
        assert np.max(np.abs(c[b] - C)) <= 2e-6
        band_check(C, got[b], want, u, 2e-6)
        assert np.all(np.diff(got[b]) >= 0)


@pytest.mark.parametrize("P", [4096, 4100, 65536])
def test_resample_skewed_rows(P):
    """Rows whose mass sits on one or two particles: most chunks own no
    output, one chunk owns nearly all (long galloping searches), and the
    heavy particle may sit in the ragged last chunk."""
    rows = 6
    lw = np.full((rows, P), -np.inf, np.float32)
    lw[0, 0] = 0.0                         # one-hot at the start
    lw[1, P - 1] = 0.0                     # one-hot at the end (ragged tail when P % 4096)
    lw[2, P // 3] = 0.0                    # one-hot in the middle
    lw[3, 5], lw[3, P - 7] = 0.0, -1.0     # two heavy particles far apart
    lw[4] = workloads.resample_logw(rows=1, P=P, seed=7)[0] * 4.0  # very skewed N(0, 8^2)
    lw[5, ::97] = 0.0                      # sparse equal weights
    out = torch.empty((rows, P), dtype=torch.int32, device="cuda")
    cdf = torch.empty((rows, P), dtype=torch.float32, device="cuda")
    per.per_resample(dev(lw), 3, 7, out, out_cdf=cdf)
    got, c = host(out), host(cdf)
    for b in range(rows):
        U = oracle.u01_closed_open(3, 7, b)
        assert np.array_equal(got[b], oracle.resample_row_on_cdf(c[b], U)), f"row {b}"
        assert np.all(np.diff(got[b]) >= 0)
        assert got[b].min() >= 0 and got[b].max() < P


@pytest.mark.parametrize("P", [5 * 4096 + 100, 65536])
def test_resample_mass_at_segment_edges(P):
    """A row is split into contiguous runs of whole 4096-particle chunks
    (up to four runs, scanned side by side): mass right before, right
    after and straddling the run edges, and runs that own no mass at all,
    must give the same outputs as one scan over the row."""
    seg = ((P + 4095) // 4096 + 3) // 4 * 4096
    rows = 5
    lw = np.full((rows, P), -np.inf, np.float32)
    lw[0, seg - 1] = 0.0                            # last particle of the first run
    lw[1, seg] = 0.0                                # first particle of the second run
    lw[2, 2 * seg - 1], lw[2, 2 * seg] = 0.0, 0.0   # straddling the second edge
    lw[3, seg - 2:seg + 2] = [0.0, -0.5, -1.0, -2.0]
    lw[3, P - 1] = -3.0                             # the last particle too
    lw[4] = workloads.resample_logw(rows=1, P=P, seed=17)[0]
    lw[4, :seg] = -np.inf                           # the first run owns nothing
    out = torch.empty((rows, P), dtype=torch.int32, device="cuda")
    cdf = torch.empty((rows, P), dtype=torch.float32, device="cuda")
    per.per_resample(dev(lw), 4, 11, out, out_cdf=cdf)
    got, c = host(out), host(cdf)
    for b in range(rows):
        U = oracle.u01_closed_open(4, 11, b)
        assert np.array_equal(got[b], oracle.resample_row_on_cdf(c[b], U)), f"row {b}"
        want, C, u = oracle.resample_row(lw[b], U)
        assert np.max(np.abs(c[b] - C)) <= 2e-6
        band_check(C, got[b], want, u, 2e-6)
        assert np.all(np.diff(got[b]) >= 0)


def test_resample_equal_weights_identity_and_u_override():
    rows, P = 2, 4096
    lw = np.zeros((rows, P), np.float32)
    u = np.array([0.25, 0.75], np.float32)
    out = torch.empty((rows, P), dtype=torch.int32, device="cuda")
    per.per_resample(dev(lw), 0, 0, out, u_rows=dev(u))
    got = host(out)
    for b in range(rows):
        assert np.array_equal(got[b], np.arange(P))


# ------------------------------------------------------------ statuses ------

def test_argument_errors_raise_before_launch():
    ctx = per.PerContext(100, 0.6, SCAN)
    with pytest.raises(per.PerError) as e:
        per.per_build_cdf(ctx.handle)  # size 0
    assert e.value.code == 5
    with pytest.raises(per.PerError) as e:
        per.per_sample(ctx.handle, 10, 0, 0, TREE, torch.empty(10, dtype=torch.int32, device="cuda"))
    assert e.value.code == 6
    with pytest.raises(per.PerError):
        per.per_set_size(ctx.handle, 101)


def test_negative_priority_is_reported():
    p = np.ones(1000, np.float32)
    p[500] = -1.0
    ctx = make_ctx(p, 1.0, SCAN)
    per.per_build_cdf(ctx.handle)
    assert per.per_check(ctx.handle) == 8  # PER_ERR_VALUE
    assert per.per_check(ctx.handle) == 0  # cleared


# ---------------------------------------------------- i.i.d. tree sampling ---

@pytest.mark.parametrize("cap,B", [(1 << 19, 1024), (4096, 1), (1000, 65536)])
def test_tree_iid_sampling_matches_oracle(cap, B):
    """mode PER_TREE | PER_IID: thresholds U_k * T, one per sample (foxhunt
    "CUDA Kernels"); indices bit-exact against the oracle's descent of the
    GPU's own tree, with Philox draws and with a u01 override."""
    p = workloads.lognormal(cap, workloads.rng(120, cap))
    ctx = make_ctx(p, 0.6, TREE)
    tree = host(per.read_tree(ctx.handle))
    out = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, 13, 77, TREE | per.PER_IID, out)
    want, u = oracle.sample_tree(tree, B, 13, 77, iid=True)
    assert np.array_equal(host(out), want)
    assert np.all(p[host(out)] > 0)
    U = workloads.uniform_open_closed(B, workloads.rng(121, B))
    per.per_sample(ctx.handle, B, 0, 0, TREE | per.PER_IID, out, u01=dev(U))
    assert np.array_equal(host(out), oracle.sample_tree(tree, B, 0, 0, u01=U, iid=True)[0])
    with pytest.raises(per.PerError):
        per.per_sample(ctx.handle, B, 0, 0, SCAN | per.PER_IID, out)
    assert per.per_check(ctx.handle) == 0


# ------------------------------------------------ particle-filter resample step ---

@pytest.mark.parametrize("rows,P,D", [(4, 1024, 4), (3, 4100, 3), (2, 65536, 8), (5, 256, 1)])
def test_resample_step_gathers_states_and_resets_weights(rows, P, D):
    """per_resample_step: the indices of per_resample, the states gathered
    along the particle axis and the log-weights reset to -log P, bit for bit
    against the oracle; the reset may be done in place."""
    lw = workloads.resample_logw(rows=rows, P=P, seed=140 + D)
    g = workloads.rng(141, P * D)
    state = g.standard_normal((rows, P, D)).astype(np.float32)
    d_lw, d_state = dev(lw), dev(state)
    idx = torch.empty((rows, P), dtype=torch.int32, device="cuda")
    out_state = torch.empty((rows, P, D), dtype=torch.float32, device="cuda")
    out_lw = torch.empty((rows, P), dtype=torch.float32, device="cuda")
    per.per_resample_step(d_lw, d_state, 8, 2, idx, out_state, out_lw)
    idx2 = torch.empty((rows, P), dtype=torch.int32, device="cuda")
    cdf = torch.empty((rows, P), dtype=torch.float32, device="cuda")
    per.per_resample(d_lw, 8, 2, idx2, out_cdf=cdf)
    got_idx, c = host(idx), host(cdf)
    assert np.array_equal(got_idx, host(idx2))
    for b in range(rows):  # bit-exact: the oracle's search of the GPU's CDF
        assert np.array_equal(got_idx[b], oracle.resample_row_on_cdf(c[b], oracle.u01_closed_open(8, 2, b)))
    want_state, want_lw = oracle.resample_gather(state, got_idx)
    assert np.array_equal(host(out_state), want_state)
    assert np.array_equal(host(out_lw), want_lw)
    # in place: the log-weights themselves are reset
    per.per_resample_step(d_lw, d_state, 8, 2, idx, out_state, d_lw)
    assert np.array_equal(host(idx), got_idx)
    assert np.array_equal(host(d_lw), want_lw)

"""Pins for the CPU oracle: each test checks the oracle against something other
than itself -- cuRAND's host-side and numpy's independent Philox generators,
closed forms, exact integer / rational arithmetic, brute-force enumeration,
or values read off the pages' figures (tests/golden/).  A plausible mistake in
the oracle (a dropped term, a wrong comparison, an off-by-one in the layout, a
transposed operand) fails at least one of these.
"""
import ctypes
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- Philox ----

def _curand_host():
    """cuRAND's host-side generator library (part of the CUDA toolkit)."""
    import ctypes.util
    cands = [ctypes.util.find_library("curand"),
             os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "lib64", "libcurand.so")]
    for c in cands:
        if c:
            try:
                return ctypes.CDLL(c)
            except OSError:
                pass
    pytest.skip("cuRAND host library not available")


@pytest.mark.parametrize("seed,m,h,b", [(0x0123456789ABCDEF, 0, 0, 0), (0x0123456789ABCDEF, 3, 1, 5),
                                        (42, 0xFFFFFFFF, 0x1234, 65535), (2**64 - 1, 7, 0, 0),
                                        (12345, 2**31 + 9, 3, 777)])
def test_philox4x32_matches_curand_host_generator(seed, m, h, b):
    """cuRAND's host-side PHILOX4_32_10 generator is an independent
    implementation of the same published bijection.  For seed s it emits
    Philox4x32-10 under key (lo32(s), hi32(s)), its stream interleaving 65,536
    subsequences in counter word 2: stream position 2^18 (2^32 h + m) + 4 b
    starts the block of counter (m, h, b, 0) (a layout found by search, then
    checked here).  The oracle must give the same four words, for every
    counter word the draws use and both key words."""
    lib = _curand_host()
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # CURAND_RNG_PSEUDO_PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong((1 << 18) * ((h << 32) + m) + 4 * b)) == 0
        got = np.zeros(4, np.uint32)
        assert lib.curandGenerate(gen, got.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(4)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    want = oracle.philox4x32_10([m, h, b, 0], [seed & 0xFFFFFFFF, seed >> 32])
    assert [int(x) for x in got] == [int(x) for x in want]


@pytest.mark.parametrize("key,ctr", [
    ([0, 0], [0, 0, 0, 0]),
    ([0x243F6A8885A308D3, 0x13198A2E03707344], [0xA4093822299F31D0, 0x082EFA98EC4E6C89,
                                                0x452821E638D01377, 0xBE5466CF34E90C6C]),
    ([12345, 678], [2**64 - 3, 7, 0, 1]),
])
def test_philox4x64_matches_numpy(key, ctr):
    # numpy's Philox (an independent implementation of the same published
    # bijection) increments its 256-bit counter before producing each block.
    bg = np.random.Philox(key=np.array(key, np.uint64), counter=np.array(ctr, np.uint64))
    assert [int(x) for x in bg.state["state"]["counter"]] == ctr
    got = [int(x) for x in bg.random_raw(8)]
    c = list(ctr)
    for blk in range(2):
        # 256-bit little-endian increment
        for i in range(4):
            c[i] = (c[i] + 1) % 2**64
            if c[i] != 0:
                break
        want = [int(v) for v in oracle.philox4x64_10(c, key)]
        assert got[4 * blk:4 * blk + 4] == want


def test_philox_word_is_first_output_of_counter_offset_plus_k():
    seed, offset = 0x0123456789ABCDEF, 2**32 - 2
    for k in range(4):
        c = offset + k
        out = oracle.philox4x32_10([c & 0xFFFFFFFF, c >> 32, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
        assert oracle.philox_word(seed, offset, k) == int(out[0])


def test_u01_ranges_and_uniformity():
    n = 1 << 16
    u_oc = np.array([oracle.u01_open_closed(7, 11, k) for k in range(n)])
    u_co = np.array([oracle.u01_closed_open(7, 11, k) for k in range(n)])
    assert u_oc.min() > 0.0 and u_oc.max() <= 1.0
    assert u_co.min() >= 0.0 and u_co.max() < 1.0
    # the two share the same 24 random bits: U_oc = U_co + 2^-24 exactly
    assert np.all(u_oc - u_co == 2.0 ** -24)
    # coarse uniformity: 64 bins, chi^2 with 63 dof well inside 99.9%
    h, _ = np.histogram(u_co, bins=64, range=(0.0, 1.0))
    chi2 = ((h - n / 64) ** 2 / (n / 64)).sum()
    assert chi2 < 110.0


# ------------------------------------------------------------- CDF (scan) ---

def test_cdf_all_ones_is_index_plus_one():
    p = np.ones(100_003, np.float32)
    for alpha in (0.6, 1.0, 0.0):
        C = oracle.cdf64(p, alpha)
        assert np.array_equal(C, np.arange(1, p.size + 1, dtype=np.float64))


def test_cdf_integer_priorities_exact():
    g = np.random.default_rng(0)
    p = g.integers(0, 1000, size=5000).astype(np.float32)
    C = oracle.cdf64(p, 1.0)
    want = np.cumsum(p.astype(np.int64))
    assert np.array_equal(C, want.astype(np.float64))


def test_cdf_matches_exactly_rounded_sums():
    p = workloads.small_priorities()
    alpha = 0.6
    C = oracle.cdf64(p, alpha)
    pa = [float(x) ** alpha for x in p.astype(np.float64)]
    # spot-check prefixes against math.fsum (exactly rounded) with the serial
    # summation bound |err| <= i * 2^-53 * sum|x|
    for i in (0, 1, 17, 1000, 4095, 8191):
        exact = math.fsum(pa[: i + 1])
        assert abs(C[i] - exact) <= (i + 1) * 2.0 ** -53 * exact * 1.01 + 1e-300
    # monotone, last element is the total
    assert np.all(np.diff(C) >= 0)
    assert C[-1] == pytest.approx(math.fsum(pa), rel=1e-12)


def test_pow_alpha_special_cases():
    p = np.array([0.0, 0.25, 1.0, 4.0, 9.0], np.float32)
    assert np.array_equal(oracle.pow_alpha64(p, 0.5), np.sqrt(p.astype(np.float64)))
    assert np.array_equal(oracle.pow_alpha64(p, 1.0), p.astype(np.float64))
    # C's pow(0, 0) == 1: alpha = 0 makes every item (zeros included) weight 1
    assert np.array_equal(oracle.pow_alpha64(p, 0.0), np.ones(5))


# ------------------------------------------------------------ thresholds ----

def test_thresholds_stratified_one_per_stratum():
    # u_k = fl32(fl32(fl32(k+U)/B)*T).  With B a power of two the division is
    # exact, so the only roundings are k+U (half an ulp of k+1) and the final
    # product (half an ulp of u): the error bound below is that analysis.
    B, T = 1024, 37.25
    u = oracle.thresholds(B, seed=3, offset=100, T=T)
    assert np.all(np.diff(u.astype(np.float64)) >= 0)
    for k in range(B):
        U = oracle.u01_open_closed(3, 100, k)
        exact = (Fraction(k) + Fraction(U)) / B * Fraction(T)
        ulp_u = Fraction(np.spacing(np.float32(u[k])).item())
        ulp_a = Fraction(np.spacing(np.float32(k + 1)).item())
        bound = ulp_a / 2 / B * Fraction(T) + ulp_u / 2
        assert abs(Fraction(float(u[k])) - exact) <= bound
        # one threshold per stratum [k*T/B, (k+1)*T/B] (closed, up to the final
        # rounding: a tiny U can round k+U down to k)
        assert Fraction(k) * Fraction(T) / B - ulp_u / 2 <= Fraction(float(u[k]))
        assert Fraction(float(u[k])) <= Fraction(k + 1) * Fraction(T) / B + ulp_u / 2
    assert u[-1] <= np.float32(T)


def test_thresholds_override_equals_generated():
    B = 333
    U = np.array([oracle.u01_open_closed(9, 0, k) for k in range(B)], np.float32)
    assert np.array_equal(oracle.thresholds(B, 9, 0, 5.0), oracle.thresholds(B, 0, 0, 5.0, u01=U))


# ---------------------------------------------------------- searchsorted ----

def _linear_lower_bound(c, u):
    for i, v in enumerate(c):
        if v >= u:
            return i
    return len(c) - 1


def test_lower_bound_is_searchsorted_left_with_clamp():
    g = np.random.default_rng(5)
    c = np.sort(g.integers(0, 20, size=64)).astype(np.float32)  # many ties
    for u in np.concatenate([np.arange(-1, 22, 0.5), c]):
        want = _linear_lower_bound(c, np.float32(u))
        assert oracle.lower_bound_f32(c, u) == want
        assert oracle.lower_bound_f64(c.astype(np.float64), float(np.float32(u))) == want
    # ties resolve to the first of the tied entries; beyond the end clamps to n-1
    assert oracle.lower_bound_f32(np.array([1, 2, 2, 2, 3], np.float32), 2.0) == 1
    assert oracle.lower_bound_f32(np.array([1, 2, 3], np.float32), 3.5) == 2


def _grid_count_at_or_below(c, T):
    """Number of grid points x in [1, 2^24] whose B = 1 threshold
    fl32(x 2^-24 * T) is <= c.  The product rounds monotonically in x, so the
    set is a prefix [1, X]; X is found by bisection with each candidate's
    threshold rounded by numpy's float32 multiply (an independent IEEE
    implementation) and compared with c exactly (fp64 holds every fp32)."""
    T32 = np.float32(T)
    lo, hi = 0, 1 << 24  # invariant: thr(lo) <= c (thr(0) = 0), answer in [lo, hi]
    if float(np.float32(np.float32(hi * 2.0 ** -24) * T32)) <= c:
        return hi
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if float(np.float32(np.float32(mid * 2.0 ** -24) * T32)) <= c:
            lo = mid
        else:
            hi = mid
    return lo


def _exact_grid_counts(C):
    """Per index i, the exact number of the 2^24 grid points whose threshold
    lies in (C[i-1], C[i]] -- the interval lower_bound maps to i -- with the
    last index also taking every threshold above C[n-1] (the clamp)."""
    T = np.float32(C[-1])
    below = [_grid_count_at_or_below(float(c), T) for c in C[:-1]]
    edges = np.array([0] + below + [1 << 24], np.int64)
    return np.diff(edges)


@pytest.mark.parametrize("case", ["dyadic_alpha1", "mixed_alpha07"])
def test_brute_force_frequencies_small_n(case):
    """All 2^24 values of U = m 2^-24 (m = 1 .. 2^24, the whole range of the
    24-bit uniform in (0, 1]) for B = 1, enumerated in one oracle call: with
    B = 2^24 and every U_k = 1 the stratified threshold is
    fl32(fl32(k + 1) / 2^24 * T) = fl32((k + 1) 2^-24 T) -- exactly the B = 1
    threshold of grid point k + 1, since k + 1 <= 2^24 and the division by a
    power of two are exact.  Each index must be drawn exactly as often as the
    number of grid points whose threshold falls in its CDF interval, counted
    independently by a boundary search per index, and that count must be
    2^24 * P_i within the boundary roundings.  A zero-priority item is never
    drawn."""
    if case == "dyadic_alpha1":
        # dyadic priorities: every prefix sum is exact in fp64 and fp32, so
        # the CDF is the rational cumsum and P_i is known exactly
        p = np.array([0.5, 2.0, 0.0, 1.0, 3.0, 0.0, 0.25, 1.0, 4.0, 0.125, 1.5, 0.0, 2.5, 1.0, 0.75, 0.5],
                     np.float32)
        alpha = 1.0
    else:
        p = np.array([0.3, 2.0, 0.0, 1.7, 3.1, 0.0, 0.25, 1.0, 4.0, 0.01, 1.5, 0.0, 2.5, 1e-3, 0.75],
                     np.float32)
        alpha = 0.7
    C = oracle.cdf64(p, alpha)
    if case == "dyadic_alpha1":
        assert np.array_equal(C, np.cumsum([Fraction(float(x)) for x in p]).astype(np.float64))
    M = 1 << 24
    idx, u = oracle.sample_cdf_f64(C, M, 0, 0, u01=np.ones(M, np.float32))
    # the thresholds are the B = 1 grid thresholds, in order
    for m in (1, 2, 3, 12345, M // 2 + 7, M - 1, M):
        assert u[m - 1] == np.float32(np.float32(m * 2.0 ** -24) * np.float32(C[-1]))
    counts = np.bincount(idx, minlength=p.size)
    want = _exact_grid_counts(C)
    assert np.array_equal(counts, want)
    assert np.all(counts[p == 0] == 0)
    pa = p.astype(np.float64) ** alpha
    expect = M * pa / pa.sum()
    # one grid step of U moves the threshold by T 2^-24; each boundary's fp32
    # rounding of the threshold shifts at most a grid point or two
    assert np.all(np.abs(counts - expect) <= 2.0)
    if case == "dyadic_alpha1":
        # total = 18.125 = 145/8: index i gets 2^24 p_i / 18.125 grid points
        # up to the threshold rounding at its two boundaries
        assert float(C[-1]) == 18.125
        assert np.all(np.abs(counts - M * p.astype(np.float64) / 18.125) <= 2.0)


def test_sampling_on_equal_priorities_hits_known_indices():
    # N items of equal priority, B | N: stratum k covers items [k*N/B, (k+1)*N/B)
    N, B = 4096, 256
    C = oracle.cdf64(np.ones(N, np.float32), 1.0)
    idx, u = oracle.sample_cdf_f64(C, B, 17, 0)
    k = np.arange(B)
    assert np.all(idx >= k * (N // B)) and np.all(idx < (k + 1) * (N // B))
    # and the fp32-CDF search agrees on an exactly representable CDF
    idx32, _ = oracle.sample_cdf_f32(C.astype(np.float32), B, 17, 0)
    assert np.array_equal(idx, idx32)


# -------------------------------------------------------------- updates -----

def test_apply_updates_last_duplicate_wins():
    prio = np.zeros(8, np.float32)
    out = oracle.apply_updates(prio, [3, 1, 3, 7, 1, 3], [1, 2, 3, 4, 5, 6])
    assert out.tolist() == [0, 5, 0, 6, 0, 0, 0, 4]


# ------------------------------------------------------------ sum tree ------

def test_tree_leaves_closed_forms_and_zero_padding():
    """tree_leaves is leaf i = p_i^alpha for i < n and exactly 0 above n
    (foxhunt "Tree Layout": the capacity is rounded up to a power of two and
    the extra leaves hold nothing).  Pinned by values the mathematics fixes
    without calling pow: alpha = 1 keeps p; alpha = 1/2 on perfect squares and
    alpha = 1/4 on fourth powers give exact integer roots; alpha = 3/2 on
    powers of four and alpha = 3/4 on powers of 16 give exact powers of two;
    alpha = 0 gives 1 for every item below n, zeros included (C's
    pow(0, 0) = 1), but still 0 in the padding."""
    cap = 16
    sq = np.array([0, 1, 4, 9, 16, 25, 36, 49, 64, 81, 100, 121], np.float32)
    n = sq.size
    for alpha, want_fn in [(1.0, lambda x: x), (0.5, lambda x: np.round(np.sqrt(x)))]:
        lv = oracle.tree_leaves(sq, alpha, cap)
        assert lv.dtype == np.float32 and lv.size == cap
        assert np.array_equal(lv[:n], want_fn(sq.astype(np.float64)).astype(np.float32))
        assert np.all(lv[n:] == 0.0) and not np.any(np.signbit(lv[n:]))
    fourth = np.array([1, 16, 81, 256, 625], np.float32)
    assert np.array_equal(oracle.tree_leaves(fourth, 0.25, 8), np.array([1, 2, 3, 4, 5, 0, 0, 0], np.float32))
    pw4 = np.array([0.25, 1.0, 4.0, 16.0, 2.0 ** -20], np.float32)  # 4^k -> 8^k
    assert np.array_equal(oracle.tree_leaves(pw4, 1.5, 8),
                          np.array([0.125, 1, 8, 64, 2.0 ** -30, 0, 0, 0], np.float32))
    pw16 = np.array([16.0, 256.0, 2.0 ** -8], np.float32)  # 16^k -> 8^k
    assert np.array_equal(oracle.tree_leaves(pw16, 0.75, 4), np.array([8, 64, 2.0 ** -6, 0], np.float32))
    # alpha = 0: ones below n (the zero item too), zeros above
    z = np.array([0.0, 3.0, 0.0, 7.5, 1e-30], np.float32)
    lv = oracle.tree_leaves(z, 0.0, 8)
    assert np.array_equal(lv, np.array([1, 1, 1, 1, 1, 0, 0, 0], np.float32))
    # n = cap (no padding) and n = 0 (all padding)
    assert np.array_equal(oracle.tree_leaves(np.full(8, 9.0, np.float32), 0.5, 8), np.full(8, 3.0, np.float32))
    assert np.array_equal(oracle.tree_leaves(np.zeros(0, np.float32), 0.0, 8), np.zeros(8, np.float32))
    # a generic alpha: the leaf is the power rounded to fp32, so it lies
    # within about half an fp32 ulp of the exact 2^(alpha e) (60-digit mpmath)
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    e = np.arange(-30, 31, 3)
    x = (2.0 ** e).astype(np.float32)
    lv = oracle.tree_leaves(x, 0.6, 32)
    for k, v in zip(e, lv[:e.size]):
        exact = mpmath.power(2, mpmath.mpf(0.6) * int(k))  # the fp64 alpha the oracle receives
        assert abs(mpmath.mpf(float(v)) - exact) <= 0.5001 * float(np.spacing(v))
    assert np.all(lv[e.size:] == 0.0)


def _golden_layout():
    children, leaves, cap, root = {}, {}, None, None
    with open(os.path.join(GOLDEN, "segtree_layout_cap8.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            if line.startswith("capacity"):
                cap = int(line.split()[1])
            elif line.startswith("root"):
                root = int(line.split()[1])
            elif line.startswith("leaf"):
                a, b = line[4:].split(":")
                leaves[int(a)] = int(b)
            else:
                a, b = line.split(":")
                children[int(a)] = tuple(int(x) for x in b.split())
    return cap, root, children, leaves


def test_tree_layout_matches_design_doc_figure():
    cap, root, children, leaves = _golden_layout()
    for i in range(cap):
        e = np.zeros(cap, np.float32)
        e[i] = 1.0
        t = oracle.tree_build(e)
        assert t[leaves[i]] == 1.0
        # the nodes holding 1 are exactly leaf i's ancestors in the figure
        path, node = {leaves[i]}, leaves[i]
        while node != root:
            node = next(j for j, ch in children.items() if node in ch)
            path.add(node)
        assert set(np.nonzero(t[1:])[0] + 1) == path
        assert t[0] == 0.0


def test_tree_all_ones_depth_sums():
    k = 12
    t = oracle.tree_build(np.ones(1 << k, np.float32))
    for d in range(k + 1):
        assert np.all(t[1 << d: 1 << (d + 1)] == float(1 << (k - d)))


def test_tree_integer_leaves_descent_equals_exact_search():
    g = np.random.default_rng(11)
    cap = 1 << 10
    leaves = g.integers(0, 50, size=cap).astype(np.float32)
    leaves[g.choice(cap, 200, replace=False)] = 0.0
    t = oracle.tree_build(leaves)
    prefix = np.cumsum(leaves.astype(np.int64))
    assert t[1] == float(prefix[-1])
    # every integer and half-integer threshold in (0, total]
    for u2 in range(1, 2 * int(prefix[-1]) + 1):
        u = u2 / 2.0
        want = int(np.searchsorted(prefix, u, side="left"))
        assert oracle.tree_descend(t, u) == want
        assert leaves[want] > 0


def test_tree_guard_avoids_zero_subtree_after_rounding():
    # root = RN(1 + 1.5*2^-24) = 1 + 2^-23 exceeds the exact leaf sum; u = root
    # goes right, the remainder 2^-23 exceeds leaf 2's value, and the only
    # other leaf below is zero: the guard takes leaf 2, never the empty leaf 3.
    leaves = np.array([1.0, 0.0, 1.5 * 2.0 ** -24, 0.0], np.float32)
    t = oracle.tree_build(leaves)
    assert t[1] == np.float32(1.0 + 2.0 ** -23)
    assert oracle.tree_descend(t, t[1]) == 2
    # the CDF path picks the same item for the same threshold
    c = np.cumsum(leaves).astype(np.float32)
    assert oracle.lower_bound_f32(c, t[1]) in (2, 3) and leaves[2] > 0


def test_tree_random_leaves_against_fp64_search():
    p = workloads.heavy_priorities(N=1 << 14)
    cap = 1 << 14
    leaves = oracle.tree_leaves(p, 0.7, cap)
    t = oracle.tree_build(leaves)
    assert t[1] == pytest.approx(math.fsum(leaves.astype(np.float64)), rel=1e-6)
    C = np.cumsum(leaves.astype(np.float64))
    idx, u = oracle.sample_tree(t, 4096, 21, 0)
    assert np.all(leaves[idx] > 0)
    ref = np.searchsorted(C, u.astype(np.float64), side="left")
    bad = np.nonzero(idx != ref)[0]
    # disagreements only where the threshold sits within 2e-6*total of a boundary
    for k in bad:
        lo, hi = sorted((idx[k], ref[k]))
        gap = np.min(np.abs(C[lo:hi + 1] - float(u[k])))
        assert gap <= 2e-6 * C[-1]
    assert len(bad) <= 5


def test_tree_iid_closed_forms():
    """i.i.d. thresholds u_k = fl32(U_k * T) (foxhunt "CUDA Kernels"):
    all-ones leaves with U_k = (k + 1/2)/B give u_k = k + 1/2 and leaf k;
    U = 1 gives u = T and the last non-zero leaf; the smallest Philox U
    (2^-24) gives the first non-zero leaf."""
    cap = 1024
    t = oracle.tree_build(np.ones(cap, np.float32))
    B = cap
    U = ((np.arange(B) + 0.5) / B).astype(np.float32)
    u = oracle.thresholds_iid(B, 0, 0, float(t[1]), u01=U)
    assert np.array_equal(u, (np.arange(B) + 0.5).astype(np.float32))
    idx, _ = oracle.sample_tree(t, B, 0, 0, u01=U, iid=True)
    assert np.array_equal(idx, np.arange(B))
    leaves = np.zeros(cap, np.float32)
    leaves[[3, 100, 700]] = [2.0, 5.0, 1.0]
    t = oracle.tree_build(leaves)
    ends = np.array([1.0, 2.0 ** -24], np.float32)
    idx, u = oracle.sample_tree(t, 2, 0, 0, u01=ends, iid=True)
    assert u[0] == t[1] and idx.tolist() == [700, 3]


def test_tree_iid_thresholds_are_uniform_over_the_total():
    """Philox i.i.d. thresholds lie in (0, T], are not sorted, and the
    sampled frequencies match p_i / total (65,536 draws, 5 sigma)."""
    leaves = np.array([1.0, 3.0, 0.0, 6.0, 2.0, 0.0, 4.0, 8.0], np.float32)
    t = oracle.tree_build(leaves)
    B = 1 << 16
    idx, u = oracle.sample_tree(t, B, 42, 7, iid=True)
    assert np.all(u > 0) and np.all(u <= t[1])
    assert np.any(np.diff(u) < 0)
    assert np.all(leaves[idx] > 0)
    p = leaves / leaves.sum()
    freq = np.bincount(idx, minlength=leaves.size) / B
    assert np.all(np.abs(freq - p) <= 5 * np.sqrt(p * (1 - p) / B) + 1e-12)
    # stratified thresholds of the same draws differ: one per stratum
    _, us = oracle.sample_tree(t, B, 42, 7)
    k = np.arange(B)
    assert np.all((us > k * t[1] / B * (1 - 1e-6)) & (us <= (k + 1) * t[1] / B * (1 + 1e-6)))


# ------------------------------------------------------------ IS weights ----

def test_is_weights_closed_forms():
    p = np.array([1.0, 4.0, 2.0, 8.0], np.float32)
    # alpha=1: w_k = (pa_min / pa_k)^beta over the batch
    w = oracle.is_weights(p, 4, 1.0, [0, 1, 3], 0.5)
    assert np.allclose(w, [1.0, 0.5, (1 / 8) ** 0.5], rtol=1e-15)
    assert oracle.is_weights(p, 4, 0.6, [1, 2, 3], 0.0).tolist() == [1.0, 1.0, 1.0]
    eq = np.full(100, 3.5, np.float32)
    assert np.all(oracle.is_weights(eq, 100, 0.6, np.arange(50), 0.7) == 1.0)
    hp = workloads.heavy_priorities(N=4096)
    idx = np.nonzero(hp > 0)[0][::7]   # sampling never draws a zero-priority item
    w = oracle.is_weights(hp, 4096, 0.7, idx, 0.4)
    assert w.max() == 1.0 and np.all(w > 0)
    pa = hp[idx].astype(np.float64) ** 0.7
    assert np.allclose(w, (pa.min() / pa) ** 0.4, rtol=1e-12)


# -------------------------------------------------------------- resample ----

def test_resample_closed_forms():
    # weights [0.1, 0.2, 0.3, 0.4] -> CDF [0.1, 0.3, 0.6, 1.0];
    # U = 0.5, P = 4: u = [0.125, 0.375, 0.625, 0.875] -> [1, 2, 3, 3]
    lw = np.log(np.array([0.1, 0.2, 0.3, 0.4])).astype(np.float32)
    idx, C, u = oracle.resample_row(lw, 0.5)
    assert idx.tolist() == [1, 2, 3, 3]
    assert u.tolist() == [0.125, 0.375, 0.625, 0.875]
    assert C[-1] == pytest.approx(1.0, abs=1e-15)
    # two particles 1:3 -> item 0 only when U/2 <= 1/4
    lw2 = np.log(np.array([1.0, 3.0])).astype(np.float32)
    assert oracle.resample_row(lw2, 0.3)[0].tolist() == [0, 1]
    assert oracle.resample_row(lw2, 0.7)[0].tolist() == [1, 1]


def test_resample_equal_weights_is_identity_and_one_hot_is_constant():
    # (U must not round j+U to an integer in fp32: for P=1024 a U below half
    # an ulp of 1023 would make u_j = j/P fall on the previous boundary.)
    P = 1024
    for U in (0.001, 0.25, 0.5, 0.999):
        assert np.array_equal(oracle.resample_row(np.full(P, -3.0, np.float32), U)[0], np.arange(P))
    lw = np.full(P, -np.inf, np.float32)
    lw[77] = 0.0
    assert np.all(oracle.resample_row(lw, 0.5)[0] == 77)


def test_resample_rows_monotone_and_match_per_row():
    lw = workloads.resample_logw(rows=3, P=4096)
    idx = oracle.resample(lw, 1, 0)
    for b in range(3):
        assert np.all(np.diff(idx[b]) >= 0)
        U = oracle.u01_closed_open(1, 0, b)
        assert np.array_equal(idx[b], oracle.resample_row(lw[b], U)[0])
        # searching the fp32-rounded CDF differs only at boundary thresholds
        _, C, u = oracle.resample_row(lw[b], U)
        on32 = oracle.resample_row_on_cdf(C.astype(np.float32), U)
        diff = np.nonzero(on32 != idx[b])[0]
        for j in diff:
            assert np.min(np.abs(C - float(u[j]))) <= 2e-6


def test_resample_gather_pins():
    """The particle filter's gather and log-weight reset: equal weights keep
    every particle in place; a one-hot row copies the hot particle
    everywhere; the reset weight is -log P rounded once to fp32."""
    rows, P, D = 3, 1024, 4
    g = workloads.rng(130, 1)
    state = g.standard_normal((rows, P, D)).astype(np.float32)
    lw = np.zeros((rows, P), np.float32)
    lw[1] = -np.inf
    lw[1, 17] = 0.0
    idx = oracle.resample(lw, 5, 9)
    assert np.array_equal(idx[0], np.arange(P)) and np.all(idx[1] == 17)
    out, nlw = oracle.resample_gather(state, idx)
    assert np.array_equal(out[0], state[0])
    assert np.array_equal(out[1], np.broadcast_to(state[1, 17], (P, D)))
    assert np.array_equal(out[2], state[2, idx[2]])
    assert np.all(nlw == np.float32(-math.log(P)))
    assert nlw[0, 0] == np.float32(-6.931471805599453)


def test_rank_order_and_priorities_pins():
    """Rank-based PER (reading of the named path): descending priority,
    ties by lower index first, -0 ranked as +0; rank priorities 1/r; with
    alpha = 1 the rank CDF's total is the harmonic number H_n."""
    p = np.array([0.5, 2.0, 0.5, -0.0, 7.0, 0.0, 2.0], np.float32)
    assert oracle.rank_order(p).tolist() == [4, 1, 6, 0, 2, 3, 5]
    g = workloads.rng(150, 1)
    x = g.permutation(1000).astype(np.float32)
    assert np.array_equal(oracle.rank_order(x), np.argsort(-x, kind="stable"))
    q = oracle.rank_priorities(5)
    assert q.tolist() == [1.0, np.float32(0.5), np.float32(1 / 3), np.float32(0.25), np.float32(0.2)]
    n = 4096
    C = oracle.cdf64(oracle.rank_priorities(n), 1.0)
    H = math.fsum(1.0 / k for k in range(1, n + 1))
    assert abs(C[-1] - H) <= 2.0 ** -24 * H  # each 1/k rounded once to fp32
    C0 = oracle.cdf64(oracle.rank_priorities(n), 0.0)
    assert np.array_equal(C0, np.arange(1, n + 1, dtype=np.float64))  # alpha 0: uniform over ranks

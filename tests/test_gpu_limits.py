"""GPU parity at the entry points' largest sizes, against the oracle.

  * build_cdf at n = 2^28 (1 GiB of priorities: 32,768 tiles of the
    streaming scan): within 1e-5 of the total of the fp64 prefix sums,
    monotone, last value = per_total; 2^20 samples bit-exact when the oracle
    searches the GPU's CDF;
  * the sampler at its largest batch, B = 2^24, bit-exact the same way;
  * per_resample at its largest row, P = 2^23: bit-exact on the GPU's row
    CDF, within 2e-6 of the fp64 CDF, band rule for the indices;
  * the rank sort at its largest size, n = 2^24 with heavy ties: the order
    bit-exact against the oracle's stable sort.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

per = pytest.importorskip("cdf_scan_gb300")
SCAN = per.PER_SCAN


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


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


def test_build_cdf_and_sample_at_2p28():
    n = 1 << 28
    p = workloads.uniform_open_closed(n, workloads.rng(601, 1))
    ctx = per.PerContext(n, 0.6, SCAN)
    per.per_set_priorities(ctx.handle, dev(p))
    per.per_build_cdf(ctx.handle)
    B = 1 << 20
    idx = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, 61, 0, SCAN, idx)
    c = host(per.read_cdf(ctx.handle))
    assert per.per_check(ctx.handle) == 0
    assert per.per_total_host(ctx.handle, SCAN) == c[-1]
    assert np.all(np.diff(c) >= 0)
    C = oracle.cdf64(p, 0.6)
    del p
    assert np.max(np.abs(c - C)) <= 1e-5 * C[-1]
    want, _ = oracle.sample_cdf_f32(c, B, 61, 0)
    assert np.array_equal(host(idx), want)
    ctx.close()


def test_sampler_at_the_largest_batch():
    n, B = 1 << 20, 1 << 24
    p = workloads.abs_normal(n, workloads.rng(602, 1))
    ctx = per.PerContext(n, 0.6, SCAN)
    per.per_set_priorities(ctx.handle, dev(p))
    per.per_build_cdf(ctx.handle)
    idx = torch.empty(B, dtype=torch.int32, device="cuda")
    per.per_sample(ctx.handle, B, 62, 5, SCAN, idx)
    c = host(per.read_cdf(ctx.handle))
    want, _ = oracle.sample_cdf_f32(c, B, 62, 5)
    got = host(idx)
    assert np.array_equal(got, want)
    assert np.all(np.diff(got) >= 0)
    with pytest.raises(per.PerError):
        per.per_sample(ctx.handle, B + 1, 62, 5, SCAN, torch.empty(B + 1, dtype=torch.int32, device="cuda"))
    assert per.per_check(ctx.handle) == 0
    ctx.close()


def test_resample_at_the_largest_row():
    rows, P = 2, 1 << 23
    lw = workloads.resample_logw(rows=rows, P=P, seed=603)
    out = torch.empty((rows, P), dtype=torch.int32, device="cuda")
    cdf = torch.empty((rows, P), dtype=torch.float32, device="cuda")
    per.per_resample(dev(lw), 9, 7, out, out_cdf=cdf)
    got, c = host(out), host(cdf)
    for b in range(rows):
        U = oracle.u01_closed_open(9, 7, b)
        assert np.array_equal(got[b], oracle.resample_row_on_cdf(c[b], U))
        want, C, u = oracle.resample_row(lw[b], U)
        assert np.max(np.abs(c[b] - C)) <= 2e-6
        band_check(C, got[b], want, u, 2e-6)
        assert np.all(np.diff(got[b]) >= 0)
    big = torch.empty((1, P + 4), dtype=torch.int32, device="cuda")
    with pytest.raises(per.PerError):  # beyond the largest row
        per.per_resample(torch.zeros((1, P + 4), device="cuda"), 9, 7, big)


def test_rank_sort_at_the_largest_size():
    n = 1 << 24
    g = workloads.rng(604, 1)
    p = (np.round(np.abs(g.standard_normal(n)) * 64.0) / 64.0).astype(np.float32)  # heavy ties
    ctx = per.PerContext(n, 0.7, per.PER_RANK)
    per.per_set_priorities(ctx.handle, dev(p))
    per.per_rank_build(ctx.handle)
    assert np.array_equal(host(per.read_rank_order(ctx.handle)), oracle.rank_order(p))
    c = host(per.read_rank_cdf(ctx.handle)).astype(np.float64)
    C = oracle.cdf64(oracle.rank_priorities(n), 0.7)
    assert np.max(np.abs(c - C)) <= 1e-5 * C[-1]
    assert per.per_check(ctx.handle) == 0
    ctx.close()

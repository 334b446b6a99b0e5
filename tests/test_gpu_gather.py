"""GPU tests of the transition copy: per_gather and per_step_gather.

The copy has a plain definition, out[k] = rows[idx[k]], so the bar is
bit-exact equality with the host's indexing of the same rows by the same
indices; the indices and weights of per_step_gather must equal per_step's
bit for bit (they are checked against the oracle by the step tests).
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

per = pytest.importorskip("cdf_scan_gb300")
SCAN, TREE = per.PER_SCAN, per.PER_TREE


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def make_ctx(p, alpha, flags):
    ctx = per.PerContext(p.size, alpha, flags)
    per.per_set_priorities(ctx.handle, dev(p))
    return ctx


@pytest.mark.parametrize("cap,row_floats,B", [(1000, 4, 1), (1000, 12, 33), (65_536, 64, 8192),
                                              (4096, 260, 1000), (200_000, 16, 70_000)])
def test_gather_rows_equal_host_indexing(cap, row_floats, B):
    g = workloads.rng(401, cap + B)
    rows = g.standard_normal((cap, row_floats)).astype(np.float32)
    idx = g.integers(0, cap, B).astype(np.int32)
    idx[: B // 3] = idx[0]  # duplicates
    ctx = make_ctx(np.ones(cap, np.float32), 1.0, SCAN)
    out = torch.full((B, row_floats), np.nan, dtype=torch.float32, device="cuda")
    per.per_gather(ctx.handle, dev(rows), dev(idx), out)
    assert np.array_equal(host(out), rows[idx])
    assert per.per_check(ctx.handle) == 0


def test_gather_other_dtypes_and_bad_index():
    cap, B = 5000, 700
    g = workloads.rng(402)
    rows = g.integers(0, 255, (cap, 48)).astype(np.uint8)  # 48-byte rows
    idx = g.integers(0, cap, B).astype(np.int32)
    ctx = make_ctx(np.ones(cap, np.float32), 1.0, SCAN)
    out = torch.zeros((B, 48), dtype=torch.uint8, device="cuda")
    per.per_gather(ctx.handle, dev(rows), dev(idx), out)
    assert np.array_equal(host(out), rows[idx])
    assert per.per_check(ctx.handle) == 0
    bad = idx.copy()
    bad[5] = cap  # out of range: flagged, its row left as it was
    out2 = torch.zeros((B, 48), dtype=torch.uint8, device="cuda")
    per.per_gather(ctx.handle, dev(rows), dev(bad), out2)
    got = host(out2)
    assert per.per_check(ctx.handle) == 8  # PER_ERR_VALUE
    assert np.all(got[5] == 0)
    keep = np.arange(B) != 5
    assert np.array_equal(got[keep], rows[bad[keep]])
    with pytest.raises(per.PerError):  # 20-byte rows: not a multiple of 16
        per.per_gather(ctx.handle, dev(np.zeros((cap, 5), np.float32)), dev(idx),
                       torch.zeros((B, 5), dtype=torch.float32, device="cuda"))


@pytest.mark.parametrize("flags,mode,N,B,row_floats",
                         [(SCAN, SCAN, 262_144, 8192, 64),   # fused path: the copy inside the step's launch
                          (SCAN, SCAN, 50_000, 4096, 4),
                          (SCAN, SCAN, 1 << 20, 8192, 16),   # beyond the fused path: separate launches
                          (TREE, TREE, 100_000, 1024, 32),
                          (per.PER_RANK, per.PER_RANK, 100_000, 2048, 8)])
def test_step_gather_equals_step_then_host_indexing(flags, mode, N, B, row_floats):
    p = workloads.minibatch_priorities(N=N)
    g = workloads.rng(403, N)
    rows = g.standard_normal((N, row_floats)).astype(np.float32)
    d_rows = dev(rows)
    a = make_ctx(p, 0.6, flags)
    b = make_ctx(p, 0.6, flags)
    if flags == per.PER_RANK:
        per.per_rank_build(a.handle)
        per.per_rank_build(b.handle)
    ia = torch.empty(B, dtype=torch.int32, device="cuda")
    ib = torch.empty(B, dtype=torch.int32, device="cuda")
    wa = torch.empty(B, dtype=torch.float32, device="cuda")
    wb = torch.empty(B, dtype=torch.float32, device="cuda")
    out_rows = torch.full((B, row_floats), np.nan, dtype=torch.float32, device="cuda")
    for step in range(3):
        upd = dev(g.integers(0, N, B).astype(np.int32))
        newp = dev(workloads.abs_normal(B, g))
        per.per_step(a.handle, upd, newp, B, 17, step * B, mode, 0.4, ia, wa)
        per.per_step_gather(b.handle, upd, newp, B, 17, step * B, mode, 0.4, ib, wb, d_rows, out_rows)
        got_i = host(ib)
        assert np.array_equal(got_i, host(ia))
        assert np.array_equal(host(wb), host(wa))
        assert np.array_equal(host(out_rows), rows[got_i])
    assert per.per_check(a.handle) == 0
    assert per.per_check(b.handle) == 0

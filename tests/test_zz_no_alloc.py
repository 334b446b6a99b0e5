"""The allocation-free build_cdf entry point (per_build_cdf_noalloc).

Some callers cannot call cudaMalloc (they run inside a host application that
owns all device memory, or in a loop that cannot afford cudaMalloc's implicit
device synchronisation).  For them the library offers a context-free
build_cdf whose scratch is a fixed array compiled into the library.  This test
calls it through the C ABI several times in a row, on different inputs and
sizes -- one item, the one-wave and streaming kernels, and the largest size the
array allows, with and without a status word -- and checks each result
against the CPU oracle's fp64 CDF (2e-6 of the total up to 2^20 items, 1e-5
above, the tolerances of the other tests) and against the context-based
per_build_cdf, which runs the same deterministic kernels, so the two must be
identical.  The file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

per = pytest.importorskip("cdf_scan_gb300")


def reference_cdf(p, alpha):
    ctx = per.PerContext(p.size, alpha, per.PER_SCAN)
    per.per_set_priorities(ctx.handle, torch.from_numpy(p).cuda())
    per.per_build_cdf(ctx.handle)
    c = per.read_cdf(ctx.handle).cpu().numpy()[:p.size]
    assert per.per_check(ctx.handle) == 0
    ctx.close()
    return c


def test_no_alloc_build_cdf_matches_oracle_and_context_path():
    lib = per.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # (n, alpha, seed, pass a status word)
    cases = [(262144, 0.6, 301, True), (3 * 1024 * 1024 + 7, 0.7, 302, True), (1, 0.6, 303, False),
             (1 << 24, 0.6, 304, False), (262144, 0.6, 305, True)]
    for n, alpha, seed, with_status in cases:
        p = workloads.abs_normal(n, workloads.rng(seed))
        dp = torch.from_numpy(p).cuda()
        out = torch.full((n,), -1.0, dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda") if with_status else None
        rc = lib.per_build_cdf_noalloc(ctypes.c_void_p(dp.data_ptr()), n, ctypes.c_float(alpha),
                                       ctypes.c_void_p(out.data_ptr()),
                                       ctypes.c_void_p(status.data_ptr()) if with_status else None, stream)
        assert rc == 0, per.per_status_str(rc)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        if with_status:
            assert int(status.item()) == 0
        C = oracle.cdf64(p, alpha)
        tol = 2e-6 if n <= (1 << 20) else 1e-5
        assert np.all(np.diff(got) >= 0)
        assert np.max(np.abs(got - C)) <= tol * C[-1], f"n={n}"
        assert np.array_equal(got, reference_cdf(p, alpha)), f"n={n}"


def test_no_alloc_rejects_sizes_beyond_its_scratch():
    lib = per.lib()
    n = (1 << 24) + 1
    p = torch.ones(16, dtype=torch.float32, device="cuda")  # never read: rejected before launch
    rc = lib.per_build_cdf_noalloc(ctypes.c_void_p(p.data_ptr()), n, ctypes.c_float(0.6),
                                   ctypes.c_void_p(p.data_ptr()), None, None)
    assert rc == 1  # PER_ERR_ARG

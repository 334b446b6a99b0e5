"""CPU checks of the C ABI's argument validation: every call below carries at
least one argument that the entry point rejects before any CUDA call or
memory access (include/per.h states the limits), so the library answers
PER_ERR_ARG without a GPU.  Pointer arguments that are not the rejected one
are 16-byte-aligned stand-in addresses that are never dereferenced."""
import ctypes
import math

import pytest

PER_OK, PER_ERR_ARG = 0, 1
SCAN, TREE, RANK = 1, 2, 8
P16 = 0x10000      # a 16-byte-aligned stand-in address
P4 = 0x10004       # 4-byte aligned only


@pytest.fixture(scope="module")
def lib():
    import cdf_scan_gb300 as per
    return per.load_library(build_if_missing=True)


def create(lib, capacity, alpha, flags):
    h = ctypes.c_void_p(P16)
    code = lib.per_create(ctypes.byref(h), capacity, alpha, flags, None)
    return code, h.value


@pytest.mark.parametrize("capacity,alpha,flags", [
    (0, 0.6, SCAN),                    # capacity below 1
    ((1 << 30) + 1, 0.6, SCAN),        # capacity above 2^30
    (10, -0.5, SCAN),                  # negative alpha
    (10, math.nan, SCAN),              # NaN alpha
    (10, 2e30, SCAN),                  # alpha out of range
    (10, 0.6, 0),                      # no structure
    (10, 0.6, 16),                     # unknown flag
    (10, 0.6, RANK | SCAN),            # rank-based PER is a flag on its own
    ((1 << 24) + 1, 0.6, RANK),        # the rank sort's limit
])
def test_create_rejects_bad_arguments_and_clears_the_handle(lib, capacity, alpha, flags):
    code, h = create(lib, capacity, alpha, flags)
    assert code == PER_ERR_ARG
    assert h is None  # *out is set to NULL before the checks that follow it


def test_create_rejects_a_null_out_pointer(lib):
    assert lib.per_create(None, 10, 0.6, SCAN, None) == PER_ERR_ARG


def test_calls_on_a_null_context_are_argument_errors(lib):
    assert lib.per_set_size(None, 1) == PER_ERR_ARG
    assert lib.per_set_priorities(None, P16, 4, None) == PER_ERR_ARG
    assert lib.per_update(None, P16, P16, 4, None) == PER_ERR_ARG
    assert lib.per_build_cdf(None, None) == PER_ERR_ARG
    assert lib.per_rank_build(None, None) == PER_ERR_ARG
    assert lib.per_sample(None, 8, 1, 0, SCAN, None, P16, None) == PER_ERR_ARG
    assert lib.per_is_weights(None, P16, 8, 0.4, P16, None) == PER_ERR_ARG
    assert lib.per_sample_weighted(None, 8, 1, 0, SCAN, None, 0.4, P16, P16, None) == PER_ERR_ARG
    assert lib.per_step(None, None, None, 0, 8, 1, 0, SCAN, None, 0.4, P16, P16, None) == PER_ERR_ARG
    assert lib.per_gather(None, P16, 16, P16, 8, P16, None) == PER_ERR_ARG
    assert lib.per_total(None, SCAN, P16, None) == PER_ERR_ARG
    out = ctypes.c_float(0.0)
    assert lib.per_total_host(None, SCAN, ctypes.byref(out), None) == PER_ERR_ARG
    assert lib.per_check(None, None) == PER_ERR_ARG
    assert lib.per_debug_drop_tile(None, 0) == PER_ERR_ARG
    assert lib.per_destroy(None) == PER_OK  # destroying nothing is fine
    for acc in ("per_priorities_ptr", "per_cdf_ptr", "per_tree_ptr", "per_rank_order_ptr", "per_rank_cdf_ptr"):
        assert getattr(lib, acc)(None) is None


@pytest.mark.parametrize("rows,P,logw,out,cdf", [
    (1, 4, None, P16, None),           # null log-weights
    (1, 4, P16, None, None),           # null output
    (0, 4, P16, P16, None),            # no rows
    (1, 2, P16, P16, None),            # P below 4
    (1, 6, P16, P16, None),            # P not a multiple of 4
    (1, (1 << 23) + 4, P16, P16, None),  # P above 2^23
    (1, 8, P4, P16, None),             # misaligned log-weights
    (1, 8, P16, P4, None),             # misaligned output
    (1, 8, P16, P16, P4),              # misaligned CDF output
])
def test_resample_rejects_bad_arguments(lib, rows, P, logw, out, cdf):
    assert lib.per_resample(logw, rows, P, 1, 0, None, out, cdf, None) == PER_ERR_ARG


@pytest.mark.parametrize("D,state,ostate,olw", [
    (0, P16, P16, None),               # no state dimension
    (4097, P16, P16, None),            # state rows above 4096 floats
    (4, None, P16, None),              # null states
    (4, P16, None, None),              # null output states
    (4, P4, P16, None),                # misaligned states
    (4, P16, P16, P4),                 # misaligned log-weight output
])
def test_resample_step_rejects_bad_arguments(lib, D, state, ostate, olw):
    assert lib.per_resample_step(P16, state, 1, 8, D, 1, 0, None, P16, ostate, olw, None) == PER_ERR_ARG


@pytest.mark.parametrize("prio,n,alpha,cdf", [
    (None, 8, 0.6, P16),               # null input
    (P16, 8, 0.6, None),               # null output
    (P16, 0, 0.6, P16),                # empty
    (P16, (1 << 24) + 1, 0.6, P16),    # above the fixed scratch's 2^24 items
    (P16, 8, -1.0, P16),               # negative alpha
    (P16, 8, math.nan, P16),           # NaN alpha
    (P4, 8, 0.6, P16),                 # misaligned input
    (P16, 8, 0.6, P4),                 # misaligned output
])
def test_noalloc_build_cdf_rejects_bad_arguments(lib, prio, n, alpha, cdf):
    assert lib.per_build_cdf_noalloc(prio, n, alpha, cdf, None, None) == PER_ERR_ARG

"""Plain serial CPU oracle for proportional PER sampling -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
arm may import this package.  The CUDA library (``cdf_scan_gb300``) never
imports, links or calls it, and it imports nothing from the library: the two
share only the seeded input generators in ``workloads/``.

The arithmetic lives in ``per_oracle.c`` (serial C, fp64 unless the method
fixes fp32); this module only compiles it with gcc and marshals numpy arrays.
Each wrapper names the page and section its C function follows.

Parity pins: every function here is checked by ``tests/test_oracle.py``
against something other than itself (closed forms, exact integer sums,
brute-force enumeration, cuRAND's host-side Philox4x32-10 generator and numpy's
Philox4x64 -- two independent implementations of the published bijection).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "per_oracle.c")
_HDR = os.path.join(_HERE, "per_oracle.h")
_LIB = os.path.join(_HERE, "libper_oracle.so")
_lock = threading.Lock()
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_u32p = np.ctypeslib.ndpointer(dtype=np.uint32, flags="C_CONTIGUOUS")
_u64p = np.ctypeslib.ndpointer(dtype=np.uint64, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_u64 = ctypes.c_uint64


def build(force: bool = False) -> str:
    """Compile per_oracle.c into libper_oracle.so (gcc, no FMA contraction)."""
    with _lock:
        fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(_HDR))
        if force or not fresh:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                   "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB)
    sig = {
        "oracle_philox4x32_10": (None, [_u32p, _u32p, _u32p]),
        "oracle_philox4x64_10": (None, [_u64p, _u64p, _u64p]),
        "oracle_philox_word": (ctypes.c_uint32, [_u64, _u64, _u64]),
        "oracle_u01_open_closed": (ctypes.c_float, [_u64, _u64, _u64]),
        "oracle_u01_closed_open": (ctypes.c_float, [_u64, _u64, _u64]),
        "oracle_pow_alpha64": (None, [_f32p, _i64, ctypes.c_double, _f64p]),
        "oracle_cdf64": (None, [_f32p, _i64, ctypes.c_double, _f64p]),
        "oracle_thresholds": (None, [_i64, _u64, _u64, _vp, ctypes.c_float, _f32p]),
        "oracle_lower_bound_f32": (_i64, [_f32p, _i64, ctypes.c_float]),
        "oracle_lower_bound_f64": (_i64, [_f64p, _i64, ctypes.c_double]),
        "oracle_sample_cdf_f32": (None, [_f32p, _i64, _i64, _u64, _u64, _vp, _i32p, _f32p]),
        "oracle_sample_cdf_f64": (None, [_f64p, _i64, _i64, _u64, _u64, _vp, _i32p, _f32p]),
        "oracle_apply_updates": (None, [_f32p, _i32p, _f32p, _i64]),
        "oracle_tree_leaves": (None, [_f32p, _i64, ctypes.c_double, _i64, _f32p]),
        "oracle_tree_build": (None, [_f32p, _i64, _f32p]),
        "oracle_tree_descend": (_i64, [_f32p, _i64, ctypes.c_float]),
        "oracle_sample_tree": (None, [_f32p, _i64, _i64, _u64, _u64, _vp, ctypes.c_int, _i32p, _f32p]),
        "oracle_thresholds_iid": (None, [_i64, _u64, _u64, _vp, ctypes.c_float, _f32p]),
        "oracle_is_weights": (None, [_f32p, _i64, ctypes.c_double, _i32p, _i64, ctypes.c_double, _f64p]),
        "oracle_resample_row": (None, [_f32p, _i64, ctypes.c_float, _vp, _i32p, _vp]),
        "oracle_resample_row_on_cdf": (None, [_f32p, _i64, ctypes.c_float, _i32p]),
        "oracle_resample": (None, [_f32p, _i64, _i64, _u64, _u64, _vp, _i32p]),
        "oracle_resample_gather": (None, [_f32p, _i64, _i64, _i64, _i32p, _f32p, _vp]),
        "oracle_rank_order": (None, [_f32p, _i64, _i32p]),
        "oracle_rank_priorities": (None, [_i64, _f32p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def _opt_f32(a):
    """(keepalive, pointer) for an optional float32 array argument."""
    if a is None:
        return None, None
    a = _f32(a)
    return a, a.ctypes.data_as(ctypes.c_void_p)


# ---- Philox [PHILOX] -------------------------------------------------------

def philox4x32_10(ctr, key) -> np.ndarray:
    out = np.zeros(4, np.uint32)
    _load().oracle_philox4x32_10(np.asarray(ctr, np.uint32), np.asarray(key, np.uint32), out)
    return out


def philox4x64_10(ctr, key) -> np.ndarray:
    out = np.zeros(4, np.uint64)
    _load().oracle_philox4x64_10(np.asarray(ctr, np.uint64), np.asarray(key, np.uint64), out)
    return out


def philox_word(seed: int, offset: int, k: int) -> int:
    return int(_load().oracle_philox_word(seed, offset, k))


def u01_open_closed(seed: int, offset: int, k: int) -> float:
    return float(_load().oracle_u01_open_closed(seed, offset, k))


def u01_closed_open(seed: int, offset: int, k: int) -> float:
    return float(_load().oracle_u01_closed_open(seed, offset, k))


# ---- scan path [PR615], searchsorted [PF] ----------------------------------

def pow_alpha64(p, alpha: float) -> np.ndarray:
    p = _f32(p)
    out = np.empty(p.size, np.float64)
    _load().oracle_pow_alpha64(p, p.size, alpha, out)
    return out


def cdf64(p, alpha: float) -> np.ndarray:
    """Serial fp64 prefix sum of p**alpha."""
    p = _f32(p)
    out = np.empty(p.size, np.float64)
    _load().oracle_cdf64(p, p.size, alpha, out)
    return out


def thresholds(B: int, seed: int, offset: int, T: float, u01=None) -> np.ndarray:
    keep, ptr = _opt_f32(u01)
    out = np.empty(B, np.float32)
    _load().oracle_thresholds(B, seed, offset, ptr, np.float32(T), out)
    return out


def thresholds_iid(B: int, seed: int, offset: int, T: float, u01=None) -> np.ndarray:
    """i.i.d. thresholds u_k = fl32(U_k * T) (foxhunt "CUDA Kernels")."""
    keep, ptr = _opt_f32(u01)
    out = np.empty(B, np.float32)
    _load().oracle_thresholds_iid(B, seed, offset, ptr, np.float32(T), out)
    return out


def lower_bound_f32(c, u: float) -> int:
    c = _f32(c)
    return int(_load().oracle_lower_bound_f32(c, c.size, np.float32(u)))


def lower_bound_f64(c, u: float) -> int:
    c = np.ascontiguousarray(c, np.float64)
    return int(_load().oracle_lower_bound_f64(c, c.size, float(u)))


def sample_cdf_f32(cdf, B: int, seed: int, offset: int, u01=None):
    """Stratified sample by searching an fp32 CDF (e.g. the GPU's). -> (idx, u)"""
    cdf = _f32(cdf)
    keep, ptr = _opt_f32(u01)
    idx = np.empty(B, np.int32)
    u = np.empty(B, np.float32)
    _load().oracle_sample_cdf_f32(cdf, cdf.size, B, seed, offset, ptr, idx, u)
    return idx, u


def sample_cdf_f64(C, B: int, seed: int, offset: int, u01=None):
    """Stratified sample by searching the oracle's fp64 CDF. -> (idx, u)"""
    C = np.ascontiguousarray(C, np.float64)
    keep, ptr = _opt_f32(u01)
    idx = np.empty(B, np.int32)
    u = np.empty(B, np.float32)
    _load().oracle_sample_cdf_f64(C, C.size, B, seed, offset, ptr, idx, u)
    return idx, u


def apply_updates(prio, idx, p) -> np.ndarray:
    """Return a copy of prio with the batch applied in order (last duplicate wins)."""
    out = _f32(prio).copy()
    idx = np.ascontiguousarray(idx, np.int32)
    _load().oracle_apply_updates(out, idx, _f32(p), idx.size)
    return out


# ---- sum segment tree [SEGTREE] --------------------------------------------

def tree_leaves(p, alpha: float, cap_pow2: int) -> np.ndarray:
    p = _f32(p)
    out = np.empty(cap_pow2, np.float32)
    _load().oracle_tree_leaves(p, p.size, alpha, cap_pow2, out)
    return out


def tree_build(leaves) -> np.ndarray:
    leaves = _f32(leaves)
    cap = leaves.size
    tree = np.empty(2 * cap, np.float32)
    _load().oracle_tree_build(leaves, cap, tree)
    return tree


def tree_descend(tree, u: float) -> int:
    tree = _f32(tree)
    return int(_load().oracle_tree_descend(tree, tree.size // 2, np.float32(u)))


def sample_tree(tree, B: int, seed: int, offset: int, u01=None, iid: bool = False):
    tree = _f32(tree)
    keep, ptr = _opt_f32(u01)
    idx = np.empty(B, np.int32)
    u = np.empty(B, np.float32)
    _load().oracle_sample_tree(tree, tree.size // 2, B, seed, offset, ptr, int(iid), idx, u)
    return idx, u


# ---- importance-sampling weights -------------------------------------------

def is_weights(p, n_valid: int, alpha: float, idx, beta: float) -> np.ndarray:
    idx = np.ascontiguousarray(idx, np.int32)
    w = np.empty(idx.size, np.float64)
    _load().oracle_is_weights(_f32(p), n_valid, alpha, idx, idx.size, beta, w)
    return w


# ---- row resampling [PF] ---------------------------------------------------

def resample_row(lw, U: float):
    """-> (idx int32[P], C float64[P], u float32[P])"""
    lw = _f32(lw)
    P = lw.size
    C = np.empty(P, np.float64)
    u = np.empty(P, np.float32)
    idx = np.empty(P, np.int32)
    _load().oracle_resample_row(lw, P, np.float32(U), C.ctypes.data_as(ctypes.c_void_p), idx,
                                u.ctypes.data_as(ctypes.c_void_p))
    return idx, C, u


def resample_row_on_cdf(c, U: float) -> np.ndarray:
    c = _f32(c)
    idx = np.empty(c.size, np.int32)
    _load().oracle_resample_row_on_cdf(c, c.size, np.float32(U), idx)
    return idx


def resample(lw, seed: int, offset: int, u_rows=None) -> np.ndarray:
    lw = _f32(lw)
    rows, P = lw.shape
    keep, ptr = _opt_f32(u_rows)
    idx = np.empty((rows, P), np.int32)
    _load().oracle_resample(lw, rows, P, seed, offset, ptr, idx)
    return idx


def resample_gather(state, idx):
    """out_state[b, j] = state[b, idx[b, j]], out_logw = fl32(-log P) (the
    particle filter's gather and weight reset)."""
    state = np.ascontiguousarray(state, np.float32)
    rows, P, D = state.shape
    idx = np.ascontiguousarray(idx, np.int32)
    out = np.empty_like(state)
    lw = np.empty((rows, P), np.float32)
    _load().oracle_resample_gather(state, rows, P, D, idx, out, lw.ctypes.data_as(ctypes.c_void_p))
    return out, lw


# ---- rank-based PER --------------------------------------------------------

def rank_order(p) -> np.ndarray:
    """order[r] = item of rank r + 1 (highest priority first; ties: lower
    index first)."""
    p = _f32(p)
    order = np.empty(p.size, np.int32)
    _load().oracle_rank_order(p, p.size, order)
    return order


def rank_priorities(n: int) -> np.ndarray:
    """q[r] = fl32(1 / (r + 1)), the priority of rank r + 1."""
    q = np.empty(n, np.float32)
    _load().oracle_rank_priorities(n, q)
    return q

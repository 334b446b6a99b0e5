"""Python binding of libper_gb300.so (proportional PER sampling on GB300).

Argument marshalling only: every function has the name of the C entry point
in include/per.h, checks that tensors are CUDA tensors of the right dtype and
layout, passes ``tensor.data_ptr()`` and the current torch stream, and raises
``PerError`` on a non-OK status.  All arithmetic runs in the library's
kernels; there is no fallback: importing this module on a machine where the
library cannot be loaded raises.

PyTorch provides device memory and streams only.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

PER_OK = 0
PER_SCAN = 1
PER_TREE = 2
PER_IID = 4  # sampling-mode flag with PER_TREE: i.i.d. thresholds
PER_RANK = 8  # rank-based PER: a context flag on its own, and the sampling mode of such a context
STATUS_NAMES = {0: "PER_OK", 1: "PER_ERR_ARG", 2: "PER_ERR_CUDA", 3: "PER_ERR_OOM", 4: "PER_ERR_TIMEOUT",
                5: "PER_ERR_EMPTY", 6: "PER_ERR_STATE", 7: "PER_ERR_RANGE", 8: "PER_ERR_VALUE"}

LIB_PATH = _build.LIB

# Every entry point declared in include/per.h: name -> (restype, argtypes).
_vp, _i32, _i64, _u64, _f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_float
SIGNATURES = {
    "per_status_str": (ctypes.c_char_p, [ctypes.c_int]),
    "per_create": (ctypes.c_int, [ctypes.POINTER(_vp), _i64, _f32, ctypes.c_uint32, _vp]),
    "per_destroy": (ctypes.c_int, [_vp]),
    "per_set_size": (ctypes.c_int, [_vp, _i64]),
    "per_size": (_i64, [_vp]),
    "per_capacity_pow2": (_i64, [_vp]),
    "per_set_priorities": (ctypes.c_int, [_vp, _vp, _i64, _vp]),
    "per_update": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp]),
    "per_build_cdf": (ctypes.c_int, [_vp, _vp]),
    "per_build_cdf_noalloc": (ctypes.c_int, [_vp, _i64, _f32, _vp, _vp, _vp]),
    "per_sample": (ctypes.c_int, [_vp, _i32, _u64, _u64, ctypes.c_int, _vp, _vp, _vp]),
    "per_is_weights": (ctypes.c_int, [_vp, _vp, _i32, _f32, _vp, _vp]),
    "per_sample_weighted": (ctypes.c_int, [_vp, _i32, _u64, _u64, ctypes.c_int, _vp, _f32, _vp, _vp, _vp]),
    "per_step": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _u64, _u64, ctypes.c_int, _vp, _f32, _vp, _vp, _vp]),
    "per_gather": (ctypes.c_int, [_vp, _vp, _i64, _vp, _i32, _vp, _vp]),
    "per_step_gather": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _u64, _u64, ctypes.c_int, _vp, _f32, _vp, _vp,
                                       _vp, _i64, _vp, _vp]),
    "per_total": (ctypes.c_int, [_vp, ctypes.c_int, _vp, _vp]),
    "per_total_host": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.POINTER(_f32), _vp]),
    "per_priorities_ptr": (_vp, [_vp]),
    "per_cdf_ptr": (_vp, [_vp]),
    "per_tree_ptr": (_vp, [_vp]),
    "per_rank_build": (ctypes.c_int, [_vp, _vp]),
    "per_rank_order_ptr": (_vp, [_vp]),
    "per_rank_cdf_ptr": (_vp, [_vp]),
    "per_check": (ctypes.c_int, [_vp, _vp]),
    "per_debug_drop_tile": (ctypes.c_int, [_vp, _i64]),
    "per_resample": (ctypes.c_int, [_vp, _i32, _i32, _u64, _u64, _vp, _vp, _vp, _vp]),
    "per_resample_step": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _u64, _u64, _vp, _vp, _vp, _vp, _vp]),
    "per_launch_count": (_u64, []),
}


class PerError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}")


def load_library(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library; raise if impossible."""
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libper_gb300.so not found at {LIB_PATH}; run cdf_scan_gb300._build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load_library()
    return _lib


def _check(fn: str, code: int):
    if code != PER_OK:
        raise PerError(fn, code)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None, dtype: torch.dtype, name: str, numel: int | None = None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} holds {t.numel()} elements, needs {numel}")
    return t.data_ptr()


# ---- entry points (same names as include/per.h) ------------------------------

def per_status_str(code: int) -> str:
    return lib().per_status_str(code).decode()


def per_create(capacity: int, alpha: float, flags: int = PER_SCAN | PER_TREE, stream=None) -> int:
    h = ctypes.c_void_p()
    _check("per_create", lib().per_create(ctypes.byref(h), capacity, alpha, flags, _stream(stream)))
    return h.value


def per_destroy(ctx: int) -> None:
    _check("per_destroy", lib().per_destroy(ctx))


def per_set_size(ctx: int, n: int) -> None:
    _check("per_set_size", lib().per_set_size(ctx, n))


def per_size(ctx: int) -> int:
    return int(lib().per_size(ctx))


def per_capacity_pow2(ctx: int) -> int:
    return int(lib().per_capacity_pow2(ctx))


def per_set_priorities(ctx: int, prio: torch.Tensor, stream=None) -> None:
    _check("per_set_priorities",
           lib().per_set_priorities(ctx, _ptr(prio, torch.float32, "prio"), prio.numel(), _stream(stream)))


def per_update(ctx: int, idx: torch.Tensor, prio: torch.Tensor, stream=None) -> None:
    n = idx.numel()
    _check("per_update", lib().per_update(ctx, _ptr(idx, torch.int32, "idx"), _ptr(prio, torch.float32, "prio", n),
                                          n, _stream(stream)))


def per_build_cdf(ctx: int, stream=None) -> None:
    _check("per_build_cdf", lib().per_build_cdf(ctx, _stream(stream)))


def per_rank_build(ctx: int, stream=None) -> None:
    _check("per_rank_build", lib().per_rank_build(ctx, _stream(stream)))


def per_build_cdf_noalloc(prio: torch.Tensor, alpha: float, out_cdf: torch.Tensor,
                          status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Context-free build_cdf whose scratch is a fixed array inside the
    library (for callers that cannot allocate); n <= 2^24."""
    n = prio.numel()
    _check("per_build_cdf_noalloc", lib().per_build_cdf_noalloc(
        _ptr(prio, torch.float32, "prio"), n, alpha, _ptr(out_cdf, torch.float32, "out_cdf", n),
        _ptr(status, torch.int32, "status", 1), _stream(stream)))
    return out_cdf


def per_sample(ctx: int, B: int, seed: int, offset: int, mode: int, out_idx: torch.Tensor,
               u01: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _check("per_sample", lib().per_sample(ctx, B, seed, offset, mode, _ptr(u01, torch.float32, "u01", B),
                                          _ptr(out_idx, torch.int32, "out_idx", B), _stream(stream)))
    return out_idx


def per_is_weights(ctx: int, idx: torch.Tensor, beta: float, out_w: torch.Tensor, stream=None) -> torch.Tensor:
    B = idx.numel()
    _check("per_is_weights", lib().per_is_weights(ctx, _ptr(idx, torch.int32, "idx"), B, beta,
                                                  _ptr(out_w, torch.float32, "out_w", B), _stream(stream)))
    return out_w


def per_sample_weighted(ctx: int, B: int, seed: int, offset: int, mode: int, beta: float,
                        out_idx: torch.Tensor, out_w: torch.Tensor, u01: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    _check("per_sample_weighted", lib().per_sample_weighted(
        ctx, B, seed, offset, mode, _ptr(u01, torch.float32, "u01", B), beta,
        _ptr(out_idx, torch.int32, "out_idx", B), _ptr(out_w, torch.float32, "out_w", B), _stream(stream)))
    return out_idx


def per_step(ctx: int, upd_idx: torch.Tensor | None, upd_prio: torch.Tensor | None, B: int, seed: int,
             offset: int, mode: int, beta: float, out_idx: torch.Tensor, out_w: torch.Tensor,
             u01: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    n = 0 if upd_idx is None else upd_idx.numel()
    _check("per_step", lib().per_step(
        ctx, _ptr(upd_idx, torch.int32, "upd_idx"), _ptr(upd_prio, torch.float32, "upd_prio", n), n, B, seed,
        offset, mode, _ptr(u01, torch.float32, "u01", B), beta, _ptr(out_idx, torch.int32, "out_idx", B),
        _ptr(out_w, torch.float32, "out_w", B), _stream(stream)))
    return out_idx


def _rows(t: torch.Tensor, name: str) -> tuple[int, int]:
    """(pointer, bytes per row) of a contiguous CUDA tensor of rows (first dim = rows)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda or not t.is_contiguous() or t.dim() < 1:
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of rows")
    return t.data_ptr(), t[0].numel() * t.element_size() if t.shape[0] > 0 else 0


def per_gather(ctx: int, rows: torch.Tensor, idx: torch.Tensor, out: torch.Tensor, stream=None) -> torch.Tensor:
    """out[k] = rows[idx[k]] (rows: one row per item, any dtype, row bytes a multiple of 16)."""
    rp, rb = _rows(rows, "rows")
    op, ob = _rows(out, "out")
    if ob != rb or out.shape[0] < idx.numel() or out.dtype != rows.dtype:
        raise ValueError("out: expected rows of the same size and dtype as `rows`, one per index")
    _check("per_gather", lib().per_gather(ctx, rp, rb, _ptr(idx, torch.int32, "idx"), idx.numel(), op,
                                          _stream(stream)))
    return out


def per_step_gather(ctx: int, upd_idx: torch.Tensor | None, upd_prio: torch.Tensor | None, B: int, seed: int,
                    offset: int, mode: int, beta: float, out_idx: torch.Tensor, out_w: torch.Tensor,
                    rows: torch.Tensor, out_rows: torch.Tensor, u01: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    n = 0 if upd_idx is None else upd_idx.numel()
    rp, rb = _rows(rows, "rows")
    op, ob = _rows(out_rows, "out_rows")
    if ob != rb or out_rows.shape[0] < B or out_rows.dtype != rows.dtype:
        raise ValueError("out_rows: expected B rows of the same size and dtype as `rows`")
    _check("per_step_gather", lib().per_step_gather(
        ctx, _ptr(upd_idx, torch.int32, "upd_idx"), _ptr(upd_prio, torch.float32, "upd_prio", n), n, B, seed,
        offset, mode, _ptr(u01, torch.float32, "u01", B), beta, _ptr(out_idx, torch.int32, "out_idx", B),
        _ptr(out_w, torch.float32, "out_w", B), rp, rb, op, _stream(stream)))
    return out_idx


def per_total(ctx: int, mode: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    _check("per_total", lib().per_total(ctx, mode, _ptr(out, torch.float32, "out", 1), _stream(stream)))
    return out


def per_total_host(ctx: int, mode: int, stream=None) -> float:
    v = ctypes.c_float()
    _check("per_total_host", lib().per_total_host(ctx, mode, ctypes.byref(v), _stream(stream)))
    return float(v.value)


def per_check(ctx: int, stream=None) -> int:
    """Synchronise and return (and clear) the device status code (0 = OK)."""
    return int(lib().per_check(ctx, _stream(stream)))


def per_debug_drop_tile(ctx: int, tile: int) -> None:
    """Test-only fault injection: the next scan on ctx withholds tile
    `tile`'s carry word, so waits for it run out (PER_ERR_TIMEOUT)."""
    _check("per_debug_drop_tile", lib().per_debug_drop_tile(ctx, tile))


def per_resample(logw: torch.Tensor, seed: int, offset: int, out_idx: torch.Tensor,
                 u_rows: torch.Tensor | None = None, out_cdf: torch.Tensor | None = None,
                 stream=None) -> torch.Tensor:
    rows, P = logw.shape
    _check("per_resample", lib().per_resample(
        _ptr(logw, torch.float32, "logw"), rows, P, seed, offset, _ptr(u_rows, torch.float32, "u_rows", rows),
        _ptr(out_idx, torch.int32, "out_idx", rows * P), _ptr(out_cdf, torch.float32, "out_cdf", rows * P),
        _stream(stream)))
    return out_idx


def per_resample_step(logw: torch.Tensor, state: torch.Tensor, seed: int, offset: int, out_idx: torch.Tensor,
                      out_state: torch.Tensor, out_logw: torch.Tensor | None = None,
                      u_rows: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    rows, P = logw.shape
    D = state.shape[-1]
    if tuple(state.shape) != (rows, P, D):
        raise ValueError("state must be [rows, P, D] for logw [rows, P]")
    _check("per_resample_step", lib().per_resample_step(
        _ptr(logw, torch.float32, "logw"), _ptr(state, torch.float32, "state"), rows, P, D, seed, offset,
        _ptr(u_rows, torch.float32, "u_rows", rows), _ptr(out_idx, torch.int32, "out_idx", rows * P),
        _ptr(out_state, torch.float32, "out_state", rows * P * D), _ptr(out_logw, torch.float32, "out_logw", rows * P),
        _stream(stream)))
    return out_state


def per_launch_count() -> int:
    return int(lib().per_launch_count())


# ---- views of context-owned device buffers ----------------------------------

class _DeviceArray:
    """Zero-copy description of a context-owned float32 / int32 device buffer."""

    def __init__(self, ptr: int, n: int, typestr: str = "<f4"):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def _view(ptr: int, n: int, typestr: str = "<f4") -> torch.Tensor:
    """Copy n elements from a context-owned device pointer into a new tensor."""
    if n == 0:
        return torch.empty(0, dtype=torch.float32 if typestr == "<f4" else torch.int32, device="cuda")
    return torch.as_tensor(_DeviceArray(ptr, n, typestr), device="cuda").clone()


def read_cdf(ctx: int) -> torch.Tensor:
    return _view(lib().per_cdf_ptr(ctx), per_size(ctx))


def read_tree(ctx: int) -> torch.Tensor:
    return _view(lib().per_tree_ptr(ctx), 2 * per_capacity_pow2(ctx))


def read_rank_order(ctx: int) -> torch.Tensor:
    """order[r] = the item of rank r + 1 (PER_RANK contexts, after per_rank_build)."""
    return _view(lib().per_rank_order_ptr(ctx), per_size(ctx), "<i4")


def read_rank_cdf(ctx: int) -> torch.Tensor:
    return _view(lib().per_rank_cdf_ptr(ctx), per_size(ctx))


def read_priorities(ctx: int, n: int | None = None) -> torch.Tensor:
    return _view(lib().per_priorities_ptr(ctx), per_size(ctx) if n is None else n)


class PerContext:
    """Owns one per_ctx handle (destroyed on close / garbage collection)."""

    def __init__(self, capacity: int, alpha: float, flags: int = PER_SCAN | PER_TREE, stream=None):
        self.capacity = capacity
        self.alpha = alpha
        self.flags = flags
        self.handle = per_create(capacity, alpha, flags, stream)

    def close(self):
        if self.handle:
            per_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

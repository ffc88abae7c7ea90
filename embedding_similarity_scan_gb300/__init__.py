"""Python binding of libdseq.so — the embedding similarity scan on GB300.

Argument marshalling only: every step of both paths runs in the library's
CUDA kernels.  The names mirror the C ABI in ``include/dseq.h``:

* ``dseq_create(table)``                      -> ``Context``
* ``dseq_run(ctx, starts, L, mask=None)``     -> picks ``[B, L]`` int32
* ``dseq_run_trace(ctx, starts, L, trace_seqs, mask=None)`` -> (picks, trace)
* ``dseq_destroy(ctx)``
* ``bmu_search(X, W)``                        -> (idx ``[n]`` int32, dist ``[n]`` float32)
* ``dseq_set_option`` / ``dseq_get_option`` / ``dseq_last_stat`` / ``dseq_last_error``

Arrays may be torch tensors (CPU or CUDA) or numpy arrays; outputs are
allocated on the device of the main input (CUDA tensor in, CUDA tensor out;
host in, host out).  Calls run on the current torch CUDA stream.  If the
library is not built, importing works but every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdseq.so")

DSEQ_OK = 0
DSEQ_EINVAL = -1
DSEQ_ENONFINITE = -2
DSEQ_ENOMEM = -3
DSEQ_ELAUNCH = -4
DSEQ_ETIMEOUT = -5
DSEQ_ECUDA = -6
DSEQ_EINTERNAL = -7

_CODES = {v: k for k, v in list(globals().items()) if k.startswith("DSEQ_")}

# every extern "C" symbol declared in include/dseq.h
EXPORTS = ("dseq_create", "dseq_run", "dseq_run_trace", "dseq_destroy", "bmu_search",
           "bmu_search_noalloc", "som_update", "som_epoch", "dseq_set_option",
           "dseq_get_option", "dseq_last_stat", "dseq_last_error", "dseq_get_timeline")

_lib = None


class DseqError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_CODES.get(code, code)}: {msg}")
        self.code = code


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdseq.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built: run embedding_similarity_scan_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    lib.dseq_create.argtypes = [vp, i64, i32, ctypes.c_int, vp, ctypes.POINTER(vp)]
    lib.dseq_create.restype = ctypes.c_int
    lib.dseq_run.argtypes = [vp, vp, i32, i32, vp, vp, vp]
    lib.dseq_run.restype = ctypes.c_int
    lib.dseq_run_trace.argtypes = [vp, vp, i32, i32, vp, vp, vp, i32, vp, vp]
    lib.dseq_run_trace.restype = ctypes.c_int
    lib.dseq_get_timeline.argtypes = [vp, vp, i64, ctypes.POINTER(i32), ctypes.POINTER(i32)]
    lib.dseq_get_timeline.restype = ctypes.c_int
    lib.dseq_destroy.argtypes = [vp]
    lib.dseq_destroy.restype = None
    lib.bmu_search.argtypes = [vp, i64, vp, i64, i32, vp, vp, vp]
    lib.bmu_search.restype = ctypes.c_int
    lib.bmu_search_noalloc.argtypes = [vp, i64, vp, i64, i32, vp, vp, vp]
    lib.bmu_search_noalloc.restype = ctypes.c_int
    lib.som_update.argtypes = [vp, i64, vp, i32, i32, i32, vp, ctypes.c_double, i32, vp]
    lib.som_update.restype = ctypes.c_int
    lib.som_epoch.argtypes = [vp, i64, vp, i32, i32, i32, ctypes.c_double, i32, vp, vp, vp]
    lib.som_epoch.restype = ctypes.c_int
    lib.dseq_set_option.argtypes = [vp, ctypes.c_char_p, i64]
    lib.dseq_set_option.restype = ctypes.c_int
    lib.dseq_get_option.argtypes = [vp, ctypes.c_char_p]
    lib.dseq_get_option.restype = i64
    lib.dseq_last_stat.argtypes = [ctypes.c_char_p]
    lib.dseq_last_stat.restype = i64
    lib.dseq_last_error.argtypes = []
    lib.dseq_last_error.restype = ctypes.c_char_p
    if path == LIB_PATH:
        _lib = lib
    return lib


def _check(rc: int) -> None:
    if rc != DSEQ_OK:
        raise DseqError(rc, load().dseq_last_error().decode())


# ---------------------------------------------------------------------------
# marshalling helpers


def _is_torch(x) -> bool:
    return type(x).__module__.startswith("torch")


def _ptr(x) -> int:
    if _is_torch(x):
        assert x.is_contiguous(), "tensor must be contiguous"
        return x.data_ptr()
    return x.ctypes.data


def _stream(stream, *arrays) -> int:
    if stream is not None:
        return int(getattr(stream, "cuda_stream", stream))
    if any(_is_torch(a) and a.is_cuda for a in arrays if a is not None):
        import torch

        return int(torch.cuda.current_stream().cuda_stream)
    return 0


def _as(x, dtype_name: str):
    """Contiguous array of the given dtype, keeping its kind (torch or numpy)."""
    if _is_torch(x):
        import torch

        return x.to(getattr(torch, dtype_name)).contiguous()
    import numpy as np

    return np.ascontiguousarray(x, dtype=dtype_name)


def _empty_like_kind(ref, shape, dtype_name: str):
    if _is_torch(ref):
        import torch

        return torch.empty(shape, dtype=getattr(torch, dtype_name), device=ref.device,
                           pin_memory=(not ref.is_cuda and ref.is_pinned()))
    import numpy as np

    return np.empty(shape, dtype=dtype_name)


# ---------------------------------------------------------------------------
# the API


class Context:
    """A candidate table resident on the GPU (owns a dseq_ctx)."""

    def __init__(self, handle: int, N: int, D: int):
        self.handle = handle
        self.N, self.D = N, D

    def close(self) -> None:
        if self.handle:
            load().dseq_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def dseq_create(table, stream=None) -> Context:
    """Upload and prepare an N x D float32 candidate table."""
    lib = load()
    table = _as(table, "float32")
    N, D = int(table.shape[0]), int(table.shape[1])
    h = ctypes.c_void_p()
    _check(lib.dseq_create(_ptr(table), N, D, int(_is_torch(table) and table.is_cuda),
                           _stream(stream, table), ctypes.byref(h)))
    return Context(h.value, N, D)


def dseq_destroy(ctx: Context) -> None:
    ctx.close()


def dseq_get_timeline(ctx: Context):
    """Phase stamps and wait times [iters, grid, 12] (int64 ns) of the last
    timed run, or None."""
    import numpy as np

    lib = load()
    it, gr = ctypes.c_int32(), ctypes.c_int32()
    _check(lib.dseq_get_timeline(ctx.handle, None, 0, ctypes.byref(it), ctypes.byref(gr)))
    if it.value == 0:
        return None
    out = np.empty((it.value, gr.value, 12), np.int64)
    _check(lib.dseq_get_timeline(ctx.handle, out.ctypes.data, out.size, ctypes.byref(it),
                                 ctypes.byref(gr)))
    return out


def dseq_run(ctx: Context, starts, L: int, mask=None, picks=None, stream=None):
    """B greedy max-min sequences of L picks after their starts -> picks [B, L]."""
    lib = load()
    starts = _as(starts, "int32")
    B = int(starts.shape[0])
    if mask is not None:
        mask = _as(mask, "uint8")
    if picks is None:
        picks = _empty_like_kind(starts, (B, int(L)), "int32")
    _check(lib.dseq_run(ctx.handle, _ptr(starts), B, int(L),
                        None if mask is None else _ptr(mask), _ptr(picks),
                        _stream(stream, starts, mask, picks)))
    return picks


def dseq_run_trace(ctx: Context, starts, L: int, trace_seqs, mask=None, stream=None):
    """dseq_run plus the running minimum distances of the traced sequences
    after every fold: trace [n_trace, L, N] float32 on the GPU."""
    import torch

    lib = load()
    starts = _as(starts, "int32")
    trace_seqs = _as(trace_seqs, "int32")
    B, n_trace = int(starts.shape[0]), int(trace_seqs.shape[0])
    if mask is not None:
        mask = _as(mask, "uint8")
    picks = _empty_like_kind(starts, (B, int(L)), "int32")
    trace = torch.empty((n_trace, int(L), ctx.N), dtype=torch.float32, device="cuda")
    _check(lib.dseq_run_trace(ctx.handle, _ptr(starts), B, int(L),
                              None if mask is None else _ptr(mask), _ptr(picks),
                              _ptr(trace_seqs), n_trace, trace.data_ptr(),
                              _stream(stream, starts, mask, picks, trace)))
    return picks, trace


def bmu_search(X, W, idx=None, dist=None, stream=None):
    """Best-matching unit of every row of X (n x D) in the codebook W (M x D)."""
    lib = load()
    X = _as(X, "float32")
    W = _as(W, "float32")
    n, D = int(X.shape[0]), int(X.shape[1])
    M = int(W.shape[0])
    if int(W.shape[1]) != D:
        raise ValueError("X and W must have the same number of columns")
    if idx is None:
        idx = _empty_like_kind(X, (n,), "int32")
    if dist is None:
        dist = _empty_like_kind(X, (n,), "float32")
    _check(lib.bmu_search(_ptr(X), n, _ptr(W), M, D, _ptr(idx), _ptr(dist),
                          _stream(stream, X, W, idx, dist)))
    return idx, dist


def _codebook_inout(W, side_x: int, side_y: int, D: int):
    """W is updated in place, so it must already be contiguous float32."""
    dt = str(W.dtype).replace("torch.", "")
    if dt != "float32" or not (W.is_contiguous() if _is_torch(W) else W.flags.c_contiguous):
        raise ValueError("W must be a contiguous float32 array (it is updated in place)")
    if tuple(W.shape) != (int(side_x) * int(side_y), D):
        raise ValueError(f"W must be (side_x*side_y, D) = ({int(side_x) * int(side_y)}, {D})")
    return W


def som_update(X, bmu, W, side_x: int, side_y: int, sigma: float, radius: int, stream=None):
    """Batch-map neighbourhood update of W (side_x*side_y x D, in place) from
    the samples X (n x D) and their BMUs; returns W."""
    lib = load()
    X = _as(X, "float32")
    bmu = _as(bmu, "int32")
    n, D = int(X.shape[0]), int(X.shape[1])
    _codebook_inout(W, side_x, side_y, D)
    if int(bmu.shape[0]) != n:
        raise ValueError("bmu must have one entry per sample")
    _check(lib.som_update(_ptr(X), n, _ptr(W), int(side_x), int(side_y), D, _ptr(bmu),
                          float(sigma), int(radius), _stream(stream, X, bmu, W)))
    return W


def som_epoch(X, W, side_x: int, side_y: int, sigma: float, radius: int, bmu=None, dist=None,
              stream=None):
    """One SOM epoch: BMU search of X against W, then the neighbourhood update
    of W in place.  Returns (bmu, dist) of the search."""
    lib = load()
    X = _as(X, "float32")
    n, D = int(X.shape[0]), int(X.shape[1])
    _codebook_inout(W, side_x, side_y, D)
    if bmu is None:
        bmu = _empty_like_kind(X, (n,), "int32")
    if dist is None:
        dist = _empty_like_kind(X, (n,), "float32")
    _check(lib.som_epoch(_ptr(X), n, _ptr(W), int(side_x), int(side_y), D, float(sigma),
                         int(radius), _ptr(bmu), _ptr(dist), _stream(stream, X, W, bmu, dist)))
    return bmu, dist


def bmu_search_noalloc(X, W, idx, dist, stream=None):
    """bmu_search into caller-provided device outputs, using the library's
    fixed scratch instead of allocating (for callers that cannot allocate
    device memory); X, W, idx and dist must be CUDA tensors."""
    lib = load()
    n, D = int(X.shape[0]), int(X.shape[1])
    _check(lib.bmu_search_noalloc(_ptr(X), n, _ptr(W), int(W.shape[0]), D, _ptr(idx),
                                  _ptr(dist), _stream(stream, X, W, idx, dist)))
    return idx, dist


def dseq_set_option(name: str, value: int, ctx: Context | None = None) -> None:
    _check(load().dseq_set_option(ctx.handle if ctx else None, name.encode(), int(value)))


def dseq_get_option(name: str, ctx: Context | None = None) -> int:
    return int(load().dseq_get_option(ctx.handle if ctx else None, name.encode()))


def dseq_last_stat(name: str) -> int:
    return int(load().dseq_last_stat(name.encode()))


def dseq_last_error() -> str:
    return load().dseq_last_error().decode()

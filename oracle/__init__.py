"""CPU oracle for the embedding similarity scan — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python
binding never import, load or call it, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, double precision, each sum in
ascending index order; OpenMP only across independent sequences or samples).
This module compiles it with gcc into ``liboracle.so`` next to the source and
wraps its entry points with numpy marshalling.  See ``oracle.c`` for the
passages each function follows.

Parity status of each function (what pins it, in ``tests/test_oracle.py``):
  row_norms, fold, argmax, dseq   -- pinned: hand-worked 4-point example,
      orthonormal table, duplicate rows, tiled == one pass for every tile
      size, brute-force farthest-first traversal on tiny tables, invariants.
  centroid_dist, dseq_centroid    -- pinned: hand-worked example where the
      centroid and max-min criteria disagree, the zero-centroid reading,
      brute force against an independent centroid routine, tiled == one pass.
  bmu, sqdist_pairs               -- pinned: codebook containing the samples,
      integer lattice codebook (BMU = nearest lattice point), duplicate
      neurons, brute force against an independent argmin on tiny inputs.
  som_update                      -- pinned: sigma = 0 gives the per-neuron
      mean of the assigned samples (independent group-by), identical samples,
      a lattice map whose closed-form means are the grid coordinates (edge
      neurons biased inward by the one-sided window), the window corner and
      just-outside weights, mirror symmetry of the grid.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=gnu11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]
_lock = threading.Lock()
_lib = None

_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u8p = np.ctypeslib.ndpointer(dtype=np.uint8, flags="C_CONTIGUOUS")


def compile_library(src: str = _SRC, out: str = _LIB, extra: list[str] | None = None) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc."""
    cmd = ["gcc", *_CFLAGS, *(extra or []), src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle if the library is missing or older than its source."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            compile_library()
    return _LIB


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    i64, i32 = ctypes.c_int64, ctypes.c_int32
    lib.oracle_threads.argtypes = [ctypes.c_int]
    lib.oracle_threads.restype = ctypes.c_int
    lib.oracle_row_norms.argtypes = [_f32p, i64, i32, _f64p]
    lib.oracle_row_norms.restype = None
    lib.oracle_fold.argtypes = [_f32p, i64, i32, _f64p, i64, _f64p]
    lib.oracle_fold.restype = None
    lib.oracle_fold_batch.argtypes = [_f32p, i64, i32, _f64p, _i64p, i32, _f64p, ctypes.c_int]
    lib.oracle_fold_batch.restype = None
    lib.oracle_argmax.argtypes = [_f64p, _u8p, i64, i64]
    lib.oracle_argmax.restype = i64
    lib.oracle_dseq.argtypes = [_f32p, i64, i32, _i32p, i32, i32, ctypes.c_void_p, i64,
                                _i32p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_dseq.restype = ctypes.c_int
    lib.oracle_centroid_dist.argtypes = [_f32p, i64, i32, _f64p, _i64p, i32, _f64p]
    lib.oracle_centroid_dist.restype = None
    lib.oracle_centroid_dist_batch.argtypes = [_f32p, i64, i32, _f64p, _i64p, i32, i32, _f64p,
                                               ctypes.c_int]
    lib.oracle_centroid_dist_batch.restype = None
    lib.oracle_dseq_centroid.argtypes = [_f32p, i64, i32, _i32p, i32, i32, ctypes.c_void_p, i64,
                                         _i32p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_dseq_centroid.restype = ctypes.c_int
    lib.oracle_bmu.argtypes = [_f32p, i64, _f32p, i64, i32, _i32p, _f64p, ctypes.c_void_p,
                               ctypes.c_int]
    lib.oracle_bmu.restype = None
    lib.oracle_sqdist_pairs.argtypes = [_f32p, _f32p, i32, _i64p, _i64p, i64, _f64p]
    lib.oracle_sqdist_pairs.restype = None
    lib.oracle_som_update.argtypes = [_f32p, i64, i32, _i32p, _f32p, i32, i32, ctypes.c_double,
                                      i32, _i64p, i64, _f64p, ctypes.c_int]
    lib.oracle_som_update.restype = None
    return lib


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the oracle library (building it first if needed).

    ``path`` loads another build of the same source (used by the tests that
    plant a mistake in a copy of the oracle to show the pins catch it)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def threads(n: int = 0, lib=None) -> int:
    """Number of OpenMP threads the oracle uses when asked for ``n`` (0 = default)."""
    return int((lib or load()).oracle_threads(int(n)))


def row_norms(E, lib=None) -> np.ndarray:
    E = _f32(E)
    out = np.empty(E.shape[0], np.float64)
    (lib or load()).oracle_row_norms(E, E.shape[0], E.shape[1], out)
    return out


def fold(E, nrm, p: int, m: np.ndarray, lib=None) -> None:
    """In place: m[c] <- min(m[c], 1 - cos(e_p, e_c)) for every row c."""
    E = _f32(E)
    (lib or load()).oracle_fold(E, E.shape[0], E.shape[1], np.ascontiguousarray(nrm, np.float64),
                                int(p), m)


def fold_batch(E, nrm, p, m: np.ndarray, threads: int = 0, lib=None) -> None:
    """In place, for each row r of m (R x N): fold pick p[r] into m[r]."""
    E = _f32(E)
    p = np.ascontiguousarray(p, np.int64)
    assert m.dtype == np.float64 and m.flags.c_contiguous and m.shape == (p.size, E.shape[0])
    (lib or load()).oracle_fold_batch(E, E.shape[0], E.shape[1],
                                      np.ascontiguousarray(nrm, np.float64), p, p.size, m,
                                      int(threads))


def argmax(m, masked, tile: int = 0, lib=None) -> int:
    """Argmax of m over unmasked candidates, tiled scan, lowest index on ties (-1: none)."""
    m = np.ascontiguousarray(m, np.float64)
    masked = np.ascontiguousarray(masked, np.uint8)
    return int((lib or load()).oracle_argmax(m, masked, m.size, int(tile)))


def dseq(E, starts, L: int, mask=None, tile: int = 0, threads: int = 0, lib=None):
    """Greedy max-min diversity sequences.

    Returns (picks int32[B, L], radius float64[B, L], status); radius[b, t] is
    the running minimum distance of pick t when it was picked."""
    E = _f32(E)
    starts = np.ascontiguousarray(starts, np.int32)
    B = starts.size
    picks = np.empty((B, L), np.int32)
    radius = np.empty((B, L), np.float64)
    mask_arr = None
    if mask is not None:
        mask_arr = np.ascontiguousarray(mask, np.uint8)
        assert mask_arr.size == E.shape[0]
    st = (lib or load()).oracle_dseq(
        E, E.shape[0], E.shape[1], starts, B, int(L),
        None if mask_arr is None else mask_arr.ctypes.data, int(tile), picks,
        radius.ctypes.data, int(threads))
    return picks, radius, int(st)


def centroid_dist(E, nrm, members, lib=None) -> np.ndarray:
    """Cosine distances of every row to the mean of the rows `members`."""
    E = _f32(E)
    members = np.ascontiguousarray(members, np.int64)
    out = np.empty(E.shape[0], np.float64)
    (lib or load()).oracle_centroid_dist(E, E.shape[0], E.shape[1],
                                         np.ascontiguousarray(nrm, np.float64), members,
                                         members.size, out)
    return out


def centroid_dist_batch(E, nrm, members, threads: int = 0, lib=None) -> np.ndarray:
    """centroid_dist for every row of members (R x n_members) -> R x N."""
    E = _f32(E)
    members = np.ascontiguousarray(members, np.int64)
    R, k = members.shape
    out = np.empty((R, E.shape[0]), np.float64)
    (lib or load()).oracle_centroid_dist_batch(E, E.shape[0], E.shape[1],
                                               np.ascontiguousarray(nrm, np.float64), members,
                                               R, k, out, int(threads))
    return out


def dseq_centroid(E, starts, L: int, mask=None, tile: int = 0, threads: int = 0, lib=None):
    """Greedy centroid-criterion sequences: (picks, radius, status) as dseq()."""
    E = _f32(E)
    starts = np.ascontiguousarray(starts, np.int32)
    B = starts.size
    picks = np.empty((B, L), np.int32)
    radius = np.empty((B, L), np.float64)
    mask_arr = None if mask is None else np.ascontiguousarray(mask, np.uint8)
    st = (lib or load()).oracle_dseq_centroid(
        E, E.shape[0], E.shape[1], starts, B, int(L),
        None if mask_arr is None else mask_arr.ctypes.data, int(tile), picks,
        radius.ctypes.data, int(threads))
    return picks, radius, int(st)


def bmu(X, W, threads: int = 0, lib=None):
    """Best-matching units: (idx int32[n], dist float64[n], second float64[n])."""
    X, W = _f32(X), _f32(W)
    assert X.shape[1] == W.shape[1]
    n = X.shape[0]
    idx = np.empty(n, np.int32)
    dist = np.empty(n, np.float64)
    second = np.empty(n, np.float64)
    (lib or load()).oracle_bmu(X, n, W, W.shape[0], X.shape[1], idx, dist, second.ctypes.data,
                               int(threads))
    return idx, dist, second


def sqdist_pairs(X, W, ii, jj, lib=None) -> np.ndarray:
    """Squared distances |X_ii[r] - W_jj[r]|^2 in the direct form."""
    X, W = _f32(X), _f32(W)
    ii = np.ascontiguousarray(ii, np.int64)
    jj = np.ascontiguousarray(jj, np.int64)
    out = np.empty(ii.size, np.float64)
    (lib or load()).oracle_sqdist_pairs(X, W, X.shape[1], ii, jj, ii.size, out)
    return out


def som_update(X, bmu, W, side_x: int, side_y: int, sigma: float, radius: int,
               neurons=None, threads: int = 0, lib=None) -> np.ndarray:
    """Batch-map neighbourhood update: new rows (float64) of the listed
    neurons (default all M = side_x * side_y), given every sample's BMU."""
    X, W = _f32(X), _f32(W)
    n, D = X.shape
    M = int(side_x) * int(side_y)
    assert W.shape == (M, D)
    bmu = np.ascontiguousarray(bmu, np.int32)
    assert bmu.size == n
    neurons = np.arange(M, dtype=np.int64) if neurons is None else np.ascontiguousarray(neurons, np.int64)
    out = np.empty((neurons.size, D), np.float64)
    (lib or load()).oracle_som_update(X, n, D, bmu, W, int(side_x), int(side_y), float(sigma),
                                      int(radius), neurons, neurons.size, out, int(threads))
    return out

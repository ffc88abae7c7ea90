"""Parity checkers shared by the GPU tests: the CUDA results against the CPU
oracle, under the tolerances of the method's contract.

Diversity (teacher forcing): the oracle follows the GPU's picks.  At every
iteration t, for every traced sequence:
  * the GPU's running minimum equals the oracle's within 1e-5 absolute on
    every unmasked candidate, and is -inf on every masked one;
  * the GPU's pick is unmasked (so distinct from earlier picks and the
    start), and its oracle running minimum is within 1e-5 of the oracle's
    maximum over unmasked candidates.
The oracle takes its argmax in fp64 and the kernel in fp32, so equal picks
are not required where the two maxima are within that tolerance.

BMU: the GPU index equals the oracle's, except where the oracle's best two
distances differ by less than 1e-5 relative; there any neuron within that
margin of the minimum is accepted.  "Relative" is taken against
max(d_min, |x|^2 + |w|^2): the expanded form |x|^2 + |w|^2 - 2<x, w> that
the kernel evaluates carries rounding on the scale of the norms.  The GPU
distance must equal the oracle's distance to the GPU's neuron within
1e-5 * (|x|^2 + |w|^2).
"""
from __future__ import annotations

import numpy as np

import oracle

TOL = 1e-5


def check_dseq_teacher_forced(E, starts, mask, picks, trace, trace_seqs, threads=0):
    """Raise AssertionError on the first violation; returns the worst error."""
    E = np.ascontiguousarray(E, np.float32)
    N = E.shape[0]
    picks = np.asarray(picks)
    trace_seqs = np.asarray(trace_seqs, np.int64)
    R = trace_seqs.size
    L = picks.shape[1]
    nrm = oracle.row_norms(E)
    m = np.full((R, N), np.inf)
    masked = np.zeros((R, N), bool)
    if mask is not None:
        masked |= np.asarray(mask, bool)[None, :]
    st = np.asarray(starts, np.int64)[trace_seqs]
    masked[np.arange(R), st] = True
    p = st.copy()
    worst = 0.0
    rows = np.arange(R)
    for t in range(L):
        oracle.fold_batch(E, nrm, p, m, threads=threads)
        g_m = np.asarray(trace[:, t, :], np.float64)
        live = ~masked
        if live.any():
            err = np.abs(g_m - m)[live].max()
            worst = max(worst, float(err))
            assert err <= TOL, f"t={t}: running minimum differs by {err}"
        assert np.all(np.isneginf(g_m[masked])), f"t={t}: masked candidate not -inf"
        g = picks[trace_seqs, t].astype(np.int64)
        assert np.all((g >= 0) & (g < N)), f"t={t}: pick out of range"
        assert not masked[rows, g].any(), f"t={t}: masked or repeated pick"
        best = np.where(live, m, -np.inf).max(axis=1)
        gap = best - m[rows, g]
        assert np.all(gap <= TOL), f"t={t}: pick is {gap.max()} below the oracle maximum"
        masked[rows, g] = True
        p = g
    return worst


def check_centroid_teacher_forced(E, starts, mask, picks, trace, trace_seqs, threads=0):
    """Centroid criterion under teacher forcing: at every iteration the GPU's
    centroid distances equal the oracle's (centroid of the start and the
    GPU's earlier picks) within 1e-5 on unmasked rows, masked rows are -inf,
    and each pick's oracle distance is within 1e-5 of the oracle maximum."""
    E = np.ascontiguousarray(E, np.float32)
    N = E.shape[0]
    picks = np.asarray(picks)
    trace_seqs = np.asarray(trace_seqs, np.int64)
    R = trace_seqs.size
    L = picks.shape[1]
    nrm = oracle.row_norms(E)
    masked = np.zeros((R, N), bool)
    if mask is not None:
        masked |= np.asarray(mask, bool)[None, :]
    members = np.empty((R, L + 1), np.int64)
    members[:, 0] = np.asarray(starts, np.int64)[trace_seqs]
    rows = np.arange(R)
    masked[rows, members[:, 0]] = True
    worst = 0.0
    for t in range(L):
        d = oracle.centroid_dist_batch(E, nrm, members[:, :t + 1], threads=threads)
        g = np.asarray(trace[:, t, :], np.float64)
        live = ~masked
        if live.any():
            err = np.abs(g - d)[live].max()
            worst = max(worst, float(err))
            assert err <= TOL, f"t={t}: centroid distance differs by {err}"
        assert np.all(np.isneginf(g[masked])), f"t={t}: masked candidate not -inf"
        pk = picks[trace_seqs, t].astype(np.int64)
        assert np.all((pk >= 0) & (pk < N)), f"t={t}: pick out of range"
        assert not masked[rows, pk].any(), f"t={t}: masked or repeated pick"
        best = np.where(live, d, -np.inf).max(axis=1)
        gap = best - d[rows, pk]
        assert np.all(gap <= TOL), f"t={t}: pick is {gap.max()} below the oracle maximum"
        masked[rows, pk] = True
        members[:, t + 1] = pk
    return worst


def check_picks_valid(starts, mask, picks, N):
    """Every pick is in range, unmasked, never a start of its sequence, and
    distinct within its sequence."""
    picks = np.asarray(picks)
    B, L = picks.shape
    assert np.all((picks >= 0) & (picks < N))
    for b in range(B):
        row = picks[b]
        assert len(set(row.tolist())) == L, f"sequence {b} repeats a pick"
        assert starts[b] not in set(row.tolist()), f"sequence {b} picks its start"
        if mask is not None:
            assert not np.asarray(mask, bool)[row].any(), f"sequence {b} picks a masked row"


def check_bmu(X, W, sample, idx_gpu, dist_gpu, threads=0):
    """Check the GPU result on the given sample rows.  Returns counts: the
    samples checked, those whose GPU index equals the oracle's, those whose
    oracle top-2 gap falls inside the near-tie band as read here (relative to
    max(d_min, |x|^2 + |w|^2)) and inside the narrower band relative to d_min
    alone, and the samples accepted only because of the wider reading."""
    X = np.ascontiguousarray(X, np.float32)
    W = np.ascontiguousarray(W, np.float32)
    sample = np.asarray(sample, np.int64)
    Xs = X[sample]
    ig = np.asarray(idx_gpu)[sample].astype(np.int64)
    dgpu = np.asarray(dist_gpu)[sample].astype(np.float64)
    io, do, second = oracle.bmu(Xs, W, threads=threads)
    assert np.all((ig >= 0) & (ig < W.shape[0])), "BMU index out of range"
    xn = (Xs.astype(np.float64) ** 2).sum(1)
    wn = (W.astype(np.float64) ** 2).sum(1)
    d_at_g = oracle.sqdist_pairs(X, W, sample, ig)
    margin = TOL * np.maximum(do, xn + wn[io])
    exact = ig == io
    near_tie = (second - do) <= margin
    ok = exact | (near_tie & (d_at_g <= do + margin))
    bad = np.flatnonzero(~ok)
    assert bad.size == 0, (f"{bad.size} BMU index mismatches, first sample {sample[bad[0]]}: "
                           f"gpu {ig[bad[0]]} (d={d_at_g[bad[0]]}) oracle {io[bad[0]]} "
                           f"(d={do[bad[0]]}, second {second[bad[0]]})")
    derr = np.abs(dgpu - d_at_g)
    dtol = TOL * (xn + wn[ig])
    worst = int(np.argmax(derr / dtol))
    assert np.all(derr <= dtol), (f"BMU distance off by {derr[worst]} (tol {dtol[worst]}) at "
                                  f"sample {sample[worst]}")
    narrow = (second - do) <= TOL * do
    narrow_ok = exact | (narrow & (d_at_g <= do * (1.0 + TOL)))
    return {"checked": int(sample.size), "exact": int(exact.sum()),
            "in_band": int(near_tie.sum()), "in_narrow_band": int(narrow.sum()),
            "accepted_only_by_wide_band": int((~narrow_ok).sum())}

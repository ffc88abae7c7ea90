"""Pins for the CPU oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.

Each pin function returns a list of failure strings for a given build of the
oracle.  The real build must pass every pin; copies of the oracle with one
planted mistake (a flipped comparison, a wrong norm, a dropped fold, a reset
of the running max between tiles, a sign error, a dropped mask) must each fail
at least one pin, which shows the pins are not vacuous (the same idea as the
mutated-FMA check of the Metal GEMV audit, "opus_r22_gr", on the
non-vacuity of a bitwise parity suite).
"""
from __future__ import annotations

import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# independent routines (no oracle code): brute-force references


def _brute_cosine_matrix(E: np.ndarray) -> list[list[float]]:
    """All pairwise cosine distances in pure Python (math.fsum of products)."""
    rows = [[float(v) for v in r] for r in E]
    norms = [math.sqrt(math.fsum(v * v for v in r)) for r in rows]
    n = len(rows)
    return [[1.0 - math.fsum(a * b for a, b in zip(rows[i], rows[j])) / (norms[i] * norms[j])
             for j in range(n)] for i in range(n)]


def _farthest_first(dist: list[list[float]], start: int, L: int, excluded=()) -> list[int]:
    """Gonzalez's farthest-first traversal recomputed from scratch each step:
    the next point maximises its minimum distance to the chosen set."""
    chosen = [start]
    out = []
    for _ in range(L):
        best, best_c = -math.inf, -1
        for c in range(len(dist)):
            if c in chosen or c in excluded:
                continue
            r = min(dist[p][c] for p in chosen)
            if r > best:
                best, best_c = r, c
        out.append(best_c)
        chosen.append(best_c)
    return out


def _read_square4():
    table, cases = None, []
    with open(os.path.join(GOLDEN, "dseq_square4.txt")) as f:
        for line in f:
            if line.startswith("table"):
                table = np.array([[float(v) for v in tok.split(",")] for tok in line.split()[1:]],
                                 np.float32)
            elif line.startswith("case"):
                _, s, L, mask, picks, radius = line.split()
                cases.append((int(s), int(L), None if mask == "-" else [int(v) for v in
                                                                        mask.split(",")],
                              [int(v) for v in picks.split(",")],
                              [float(v) for v in radius.split(",")]))
    return table, cases


def _read_centroid_golden():
    table, out = None, {}
    with open(os.path.join(GOLDEN, "dseq_square4.txt")) as f:
        for line in f:
            if line.startswith("ctable"):
                table = np.array([[float(v) for v in tok.split(",")] for tok in line.split()[1:]],
                                 np.float32)
            elif line.startswith("maxmin"):
                _, s, L, picks = line.split()
                out["maxmin"] = (int(s), int(L), [int(v) for v in picks.split(",")])
            elif line.startswith("centroid"):
                _, s, L, picks, radius = line.split()
                out["centroid"] = (int(s), int(L), [int(v) for v in picks.split(",")],
                                   [float(v) for v in radius.split(",")])
    return table, out


def _brute_centroid(E, start, L, excluded=()):
    """Centroid criterion recomputed from scratch with math.fsum each step."""
    rows = [[float(v) for v in r] for r in E]
    norms = [math.sqrt(math.fsum(v * v for v in r)) for r in rows]
    held, out = [start], []
    for _ in range(L):
        C = [math.fsum(rows[p][k] for p in held) / len(held) for k in range(len(rows[0]))]
        cn = math.sqrt(math.fsum(v * v for v in C))
        best, best_c = -math.inf, -1
        for c in range(len(rows)):
            if c in held or c in excluded:
                continue
            d = 1.0 if cn == 0.0 else 1.0 - math.fsum(a * b for a, b in zip(C, rows[c])) / (cn * norms[c])
            if d > best:
                best, best_c = d, c
        out.append(best_c)
        held.append(best_c)
    return out


def _read_lattice():
    out = []
    with open(os.path.join(GOLDEN, "bmu_lattice.txt")) as f:
        for line in f:
            if line.startswith("sample"):
                _, x, y, j, d = line.split()
                out.append((float(x), float(y), int(j), float(d)))
    return out


def _lattice_codebook():
    return np.array([[a, b] for a in range(-3, 4) for b in range(-3, 4)], np.float32)


# --------------------------------------------------------------------------
# pins for the diversity oracle


def pins_dseq(lib) -> list[str]:
    fails: list[str] = []

    # 1. hand-worked 4-point example, and the same table with rows rescaled
    #    (cosine distance ignores row length, so nothing may change).
    table, cases = _read_square4()
    for scale in (None, np.array([2.0, 0.5, 3.0, 7.0], np.float32)):
        E = table if scale is None else table * scale[:, None]
        for s, L, mask_list, picks, radius in cases:
            mask = None
            if mask_list is not None:
                mask = np.zeros(4, np.uint8)
                mask[mask_list] = 1
            got, rad, st = oracle.dseq(E, [s], L, mask=mask, lib=lib)
            if st != 0 or got[0].tolist() != picks:
                fails.append(f"square4 start={s} scale={scale is not None}: {got[0].tolist()} != {picks}")
            elif not np.allclose(rad[0], radius, atol=1e-12):
                fails.append(f"square4 radius start={s}: {rad[0].tolist()} != {radius}")
    # exhaustion: with row 2 masked only rows 1 and 3 remain after start 0
    mask = np.zeros(4, np.uint8)
    mask[2] = 1
    _, _, st = oracle.dseq(table, [0], 3, mask=mask, lib=lib)
    if st != -1:
        fails.append("square4: exhaustion not reported")

    # 2. orthonormal table: every distance between distinct rows is exactly 1,
    #    so every pick is a tie and the picks are the ascending indices.
    N = 11
    E = np.eye(N, dtype=np.float32)
    for s in (0, 4, 10):
        for T in (0, 1, 2, 3, 5, N):
            got, rad, st = oracle.dseq(E, [s], N - 1, tile=T, lib=lib)
            want = [c for c in range(N) if c != s]
            if st != 0 or got[0].tolist() != want:
                fails.append(f"orthonormal start={s} T={T}: {got[0].tolist()}")
            elif not np.all(rad[0] == 1.0):
                fails.append(f"orthonormal radius start={s}")

    # 3. duplicate rows: rows 3 and 5 equal (never a start), row 6 equals the
    #    start row 0.  The first of {3, 5} picked must be 3; the start's
    #    duplicate has distance ~0 and comes only after every row with a
    #    positive distance.
    rng = np.random.default_rng(7)
    E = rng.standard_normal((8, 5)).astype(np.float32)
    E[5] = E[3]
    E[6] = E[0]
    got, rad, st = oracle.dseq(E, [0], 7, lib=lib)
    order = got[0].tolist()
    if st != 0 or sorted(order) != list(range(1, 8)):
        fails.append(f"duplicates: not a permutation {order}")
    else:
        if order.index(3) > order.index(5):
            fails.append(f"duplicates: 5 before 3 in {order}")
        if order[-1] != 6 and not (order[-1] == 5 and order[-2] == 6) \
                and not (order[-2] == 5 and order[-1] == 6):
            fails.append(f"duplicates: start duplicate not last {order}")
        # the duplicate of a picked row is picked only at distance ~0
        if abs(rad[0][order.index(6)]) > 1e-12:
            fails.append("duplicates: start duplicate picked at positive distance")

    # 4. associativity of max: a tiled scan equals one pass for every tile
    #    size, including a last partial tile and tiles larger than N.
    E = workloads.clustered_table(50, 8, n_centres=4, sigma=0.3, seed=3)
    st0 = [0, 17, 33, 49]
    mask = np.zeros(50, np.uint8)
    mask[[5, 6, 40]] = 1
    base, _, _ = oracle.dseq(E, st0, 20, mask=mask, tile=0, lib=lib)
    for T in (1, 2, 7, 64, 49, 50, 55):
        got, _, _ = oracle.dseq(E, st0, 20, mask=mask, tile=T, lib=lib)
        if not np.array_equal(got, base):
            fails.append(f"associativity: tile {T} differs from one pass")

    # 5. brute force: farthest-first traversal from a full distance matrix
    #    built by an independent routine, on tiny tables.
    for seed, (n, d) in enumerate([(6, 3), (9, 4), (12, 7), (12, 2)]):
        E = np.random.default_rng(100 + seed).standard_normal((n, d)).astype(np.float32)
        dist = _brute_cosine_matrix(E)
        for s in range(0, n, 3):
            want = _farthest_first(dist, s, n - 1)
            got, _, st = oracle.dseq(E, [s], n - 1, lib=lib)
            if st != 0 or got[0].tolist() != want:
                fails.append(f"brute force n={n} start={s}: {got[0].tolist()} != {want}")
        excl = {1, n - 2}
        mask = np.zeros(n, np.uint8)
        mask[list(excl)] = 1
        want = _farthest_first(dist, 0, n - 3, excluded=excl)
        got, _, st = oracle.dseq(E, [0], n - 3, mask=mask, lib=lib)
        if st != 0 or got[0].tolist() != want:
            fails.append(f"brute force masked n={n}: {got[0].tolist()} != {want}")

    # 6. invariants on a medium table, stepping the fold and argmax by hand:
    #    the running minimum never grows, the radius of successive picks never
    #    grows, picks are distinct, never masked, never the start; and the
    #    full run equals the stepped run.
    E = workloads.clustered_table(300, 16, n_centres=8, sigma=0.3, seed=5)
    nrm = oracle.row_norms(E, lib=lib)
    mask = np.zeros(300, np.uint8)
    mask[::37] = 1
    for s in (1, 150, 299):
        m = np.full(300, np.inf)
        masked = mask.copy()
        masked[s] = 1
        p, picks, radii = s, [], []
        for t in range(40):
            prev = m.copy()
            oracle.fold(E, nrm, p, m, lib=lib)
            if np.any(m > prev):
                fails.append(f"invariant: m grew at t={t}")
                break
            w = oracle.argmax(m, masked, lib=lib)
            if w < 0 or masked[w]:
                fails.append(f"invariant: masked pick {w}")
                break
            picks.append(w)
            radii.append(m[w])
            masked[w] = 1
            p = w
        if any(radii[i + 1] > radii[i] for i in range(len(radii) - 1)):
            fails.append(f"invariant: radius grew from start {s}")
        got, rad, _ = oracle.dseq(E, [s], 40, mask=mask, lib=lib)
        if got[0].tolist() != picks or not np.array_equal(rad[0], radii):
            fails.append(f"invariant: full run differs from stepped run, start {s}")
    return fails


def pins_centroid(lib) -> list[str]:
    fails: list[str] = []
    # 1. worked example where the two criteria disagree
    E, gold = _read_centroid_golden()
    s0, L, want = gold["maxmin"]
    got, _, _ = oracle.dseq(E, [s0], L, lib=lib)
    if got[0].tolist() != want:
        fails.append(f"centroid golden (max-min side): {got[0].tolist()} != {want}")
    s0, L, want, radius = gold["centroid"]
    got, rad, st = oracle.dseq_centroid(E, [s0], L, lib=lib)
    if st != 0 or got[0].tolist() != want:
        fails.append(f"centroid golden: {got[0].tolist()} != {want}")
    elif not np.allclose(rad[0], radius, atol=1e-7):
        fails.append(f"centroid golden radius: {rad[0].tolist()} != {radius}")
    # 2. the zero-centroid reading directly
    nrm = oracle.row_norms(E, lib=lib)
    d = oracle.centroid_dist(E, nrm, [0, 2], lib=lib)
    if not np.all(d == 1.0):
        fails.append(f"zero centroid distances {d.tolist()}")
    # 3. brute force on tiny random tables (no ties) and with a mask
    for seed, (n, dd) in enumerate([(7, 3), (11, 5), (12, 8)]):
        E = np.random.default_rng(300 + seed).standard_normal((n, dd)).astype(np.float32)
        for s in (0, n // 2):
            want = _brute_centroid(E, s, n - 1)
            got, _, st = oracle.dseq_centroid(E, [s], n - 1, lib=lib)
            if st != 0 or got[0].tolist() != want:
                fails.append(f"centroid brute n={n} start={s}: {got[0].tolist()} != {want}")
        mask = np.zeros(n, np.uint8)
        mask[[1, 3]] = 1
        want = _brute_centroid(E, 0, n - 3, excluded={1, 3})
        got, _, st = oracle.dseq_centroid(E, [0], n - 3, mask=mask, lib=lib)
        if st != 0 or got[0].tolist() != want:
            fails.append(f"centroid brute masked n={n}: {got[0].tolist()} != {want}")
    # 4. tiled scan == one pass
    E = workloads.clustered_table(60, 8, n_centres=4, sigma=0.3, seed=8)
    base, _, _ = oracle.dseq_centroid(E, [0, 31, 59], 25, lib=lib)
    for T in (1, 7, 59, 64):
        got, _, _ = oracle.dseq_centroid(E, [0, 31, 59], 25, tile=T, lib=lib)
        if not np.array_equal(got, base):
            fails.append(f"centroid tile {T} differs")
    return fails


# --------------------------------------------------------------------------
# pins for the BMU oracle


def pins_bmu(lib) -> list[str]:
    fails: list[str] = []

    # 1. codebook containing the samples: distance 0 at the first matching
    #    neuron; neurons 20 (= 17) and 33 (= 3) are duplicates of lower ones.
    rng = np.random.default_rng(11)
    W = rng.uniform(-1, 1, (40, 6)).astype(np.float32)
    W[20] = W[17]
    W[33] = W[3]
    X = W[[5, 17, 20, 33, 3, 39]].copy()
    idx, dist, second = oracle.bmu(X, W, lib=lib)
    if idx.tolist() != [5, 17, 17, 3, 3, 39] or np.any(dist != 0.0):
        fails.append(f"contained: {idx.tolist()} {dist.tolist()}")
    if second[1] != 0.0 or second[0] <= 0.0:
        fails.append(f"contained: second-best {second.tolist()}")

    # 2. integer lattice codebook: the BMU is the nearest grid point, exact
    #    halves go to the lower linear index.
    W = _lattice_codebook()
    cases = _read_lattice()
    X = np.array([[x, y] for x, y, _, _ in cases], np.float32)
    idx, dist, _ = oracle.bmu(X, W, lib=lib)
    for (x, y, j, d), gi, gd in zip(cases, idx, dist):
        if gi != j or abs(gd - d) > 1e-6:
            fails.append(f"lattice ({x},{y}): {gi},{gd} != {j},{d}")

    # 3. brute force against an independent argmin (numpy broadcasting,
    #    first occurrence) on tiny random inputs.
    for seed, (n, M, D) in enumerate([(7, 5, 3), (33, 64, 9), (64, 17, 64)]):
        r = np.random.default_rng(200 + seed)
        X = r.standard_normal((n, D)).astype(np.float32)
        W = r.standard_normal((M, D)).astype(np.float32)
        full = ((X[:, None, :].astype(np.float64) - W[None].astype(np.float64)) ** 2).sum(-1)
        want = full.argmin(axis=1)
        idx, dist, second = oracle.bmu(X, W, lib=lib)
        srt = np.sort(full, axis=1)
        if not np.array_equal(idx, want):
            fails.append(f"brute bmu n={n} M={M}: idx differ")
        elif not np.allclose(dist, full[np.arange(n), want], rtol=1e-12, atol=0):
            fails.append(f"brute bmu n={n} M={M}: dist differ")
        elif not np.allclose(second, srt[:, 1], rtol=1e-12, atol=0):
            fails.append(f"brute bmu n={n} M={M}: second differ")
        ii = np.repeat(np.arange(n), 2)
        jj = np.tile([0, M - 1], n)
        pairs = oracle.sqdist_pairs(X, W, ii, jj, lib=lib)
        if not np.allclose(pairs, full[ii, jj], rtol=1e-12, atol=0):
            fails.append(f"sqdist_pairs n={n} M={M} differ")
    return fails


def _read_som_golden():
    out = {"expect": []}
    with open(os.path.join(GOLDEN, "som_grid3x2.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *vals = line.split()
            if key == "sides":
                out["sides"] = (int(vals[0]), int(vals[1]))
            elif key == "sigma":
                out["sigma"] = float(vals[0])
            elif key == "samples":
                out["X"] = np.array([[float(v) for v in t.split(",")] for t in vals], np.float32)
            elif key == "bmu":
                out["bmu"] = np.array([int(v) for v in vals], np.int32)
            elif key == "old":
                out["old"] = float(vals[0])
            elif key == "expect":
                R = int(vals[0].split("=")[1])
                out["expect"].append((R, np.array([[float(v) for v in t.split(",")]
                                                    for t in vals[1:]])))
    return out


def pins_som(lib) -> list[str]:
    fails: list[str] = []

    # 0. the hand-worked 3 x 2 map
    g = _read_som_golden()
    sx, sy = g["sides"]
    W = np.full((sx * sy, g["X"].shape[1]), g["old"], np.float32)
    for R, want in g["expect"]:
        got = oracle.som_update(g["X"], g["bmu"], W, sx, sy, g["sigma"], R, lib=lib)
        if not np.allclose(got, want, rtol=0, atol=1e-12):
            fails.append(f"golden R={R}: {got.tolist()}")
    got = oracle.som_update(g["X"], g["bmu"], W, sx, sy, 0.0, 1, lib=lib)
    if not np.allclose(got, g["expect"][1][1], rtol=0, atol=1e-12):
        fails.append("golden sigma=0 differs from R=0")

    # 1. sigma = 0: each neuron is the mean of its own samples (an independent
    #    group-by); neurons without samples keep their rows.
    rng = np.random.default_rng(31)
    sx, sy, D, n = 6, 4, 5, 100
    M = sx * sy
    X = rng.standard_normal((n, D)).astype(np.float32)
    bmu = rng.integers(0, M - 5, n).astype(np.int32)  # the last five neurons get nothing
    W = rng.standard_normal((M, D)).astype(np.float32)
    sums = np.zeros((M, D))
    np.add.at(sums, bmu, X.astype(np.float64))
    cnt = np.bincount(bmu, minlength=M)
    want = np.where(cnt[:, None] > 0, sums / np.maximum(cnt, 1)[:, None], W.astype(np.float64))
    for R in (0, 3):
        got = oracle.som_update(X, bmu, W, sx, sy, 0.0, R, lib=lib)
        if not np.allclose(got, want, rtol=1e-13, atol=1e-13):
            fails.append(f"sigma=0 R={R}: not the per-neuron mean")

    # 2. identical samples: every neuron some BMU's window reaches becomes
    #    that sample; the rest keep their rows.
    x0 = rng.standard_normal(D).astype(np.float32)
    Xs = np.tile(x0, (7, 1))
    bmu = np.array([0, 0, 9, 9, 9, 23, 23], np.int32)
    got = oracle.som_update(Xs, bmu, W, sx, sy, 1.1, 1, lib=lib)
    cols, rows = np.arange(M) % sx, np.arange(M) // sx
    reach = np.zeros(M, bool)
    for c in np.unique(bmu):
        reach |= (np.abs(cols - c % sx) <= 1) & (np.abs(rows - c // sx) <= 1)
    want = np.where(reach[:, None], x0.astype(np.float64)[None, :], W.astype(np.float64))
    if not np.allclose(got, want, rtol=1e-13, atol=1e-13):
        fails.append("identical samples: wrong rows")

    # 3. lattice map, one sample per neuron holding the neuron's own grid
    #    coordinates.  The Gaussian factorises over the axes and the window is
    #    a product of intervals, so each coordinate of the new row is a 1-D
    #    weighted mean of the coordinates in the window, which for neurons at
    #    least R from every edge is the neuron's own coordinate.
    sx, sy, R, sigma = 7, 5, 2, 1.3
    M = sx * sy
    cols, rows = np.arange(M) % sx, np.arange(M) // sx
    Xl = np.stack([cols, rows], 1).astype(np.float32)
    got = oracle.som_update(Xl, np.arange(M, dtype=np.int32), np.zeros((M, 2), np.float32), sx, sy,
                            sigma, R, lib=lib)

    def mean_1d(c, side):
        ks = np.arange(max(0, c - R), min(side - 1, c + R) + 1)
        w = np.exp(-((ks - c) ** 2) / (2 * sigma * sigma))
        return float((w * ks).sum() / w.sum())

    want = np.array([[mean_1d(c, sx), mean_1d(r, sy)] for c, r in zip(cols, rows)])
    if not np.allclose(got, want, rtol=0, atol=1e-12):
        fails.append("lattice map: edge or interior means wrong")
    inner = (cols >= R) & (cols < sx - R) & (rows >= R) & (rows < sy - R)
    if not np.allclose(got[inner], Xl[inner], rtol=0, atol=1e-12):
        fails.append("lattice map: interior neurons moved")

    # 4. the window: a sample at the corner (R, R) counts with exp(-R^2 / sigma^2),
    #    one at (R + 1, 0) does not count.
    sx = sy = 9
    M = 81
    R, sigma = 2, 1.7
    j = 4 * sx + 4
    Xw = np.array([[1.0], [5.0], [1000.0]], np.float32)
    bmu = np.array([j, (4 + R) * sx + 4 + R, 4 * sx + 4 + R + 1], np.int32)
    got = oracle.som_update(Xw, bmu, np.zeros((M, 1), np.float32), sx, sy, sigma, R,
                            neurons=[j], lib=lib)
    h = np.exp(-(R * R) / (sigma * sigma))
    if abs(got[0, 0] - (1.0 + 5.0 * h) / (1.0 + h)) > 1e-12:
        fails.append(f"window corner / outside: {got[0, 0]}")

    # 5. mirror symmetry: reflecting the map's columns reflects the result.
    sx, sy, D, n = 8, 6, 3, 60
    M = sx * sy
    X = rng.standard_normal((n, D)).astype(np.float32)
    bmu = rng.integers(0, M, n).astype(np.int32)
    W = rng.standard_normal((M, D)).astype(np.float32)
    flip = (np.arange(M) // sx) * sx + (sx - 1 - np.arange(M) % sx)
    a = oracle.som_update(X, bmu, W, sx, sy, 1.4, 2, lib=lib)
    b = oracle.som_update(X, flip[bmu].astype(np.int32), W[flip], sx, sy, 1.4, 2, lib=lib)
    if not np.allclose(a[flip], b, rtol=1e-12, atol=1e-12):
        fails.append("mirror symmetry broken")
    # a subset of neurons gives the same rows as the whole map
    sub = np.array([5, 0, 47, 13])
    if not np.array_equal(oracle.som_update(X, bmu, W, sx, sy, 1.4, 2, neurons=sub, lib=lib),
                          a[sub]):
        fails.append("neuron subset differs from the whole map")
    return fails


# --------------------------------------------------------------------------


def test_dseq_pins(oracle_lib):
    assert pins_dseq(oracle_lib) == []


def test_centroid_pins(oracle_lib):
    assert pins_centroid(oracle_lib) == []


def test_som_pins(oracle_lib):
    assert pins_som(oracle_lib) == []


def test_bmu_pins(oracle_lib):
    assert pins_bmu(oracle_lib) == []


def test_threads_and_parallel_equals_serial(oracle_lib):
    assert oracle.threads(1) == 1
    E = workloads.gaussian_table(200, 12, seed=9)
    st = workloads.starts(200, 16, seed=9)
    a, ra, _ = oracle.dseq(E, st, 25, threads=1)
    b, rb, _ = oracle.dseq(E, st, 25, threads=4)
    assert np.array_equal(a, b) and np.array_equal(ra, rb)
    X = workloads.bmu_samples(50, 8, seed=1)
    W = workloads.codebook(70, 8, seed=1)
    assert all(np.array_equal(u, v) for u, v in zip(oracle.bmu(X, W, threads=1),
                                                     oracle.bmu(X, W, threads=3)))


# --------------------------------------------------------------------------
# non-vacuity: plant one mistake in a copy of the oracle, on the CPU

_SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "ties_to_highest": ("if (best_idx < 0 || m[c] > best) {",
                        "if (best_idx < 0 || m[c] >= best) {", "dseq"),
    "wrong_norm": ("return 1.0 - s / (nrm[p] * nrm[c]);",
                   "return 1.0 - s / (nrm[p] * nrm[p]);", "dseq"),
    "no_min_fold": ("if (d < m[c]) m[c] = d;", "m[c] = d;", "dseq"),
    "reset_between_tiles": ("int64_t t1 = t0 + T < N ? t0 + T : N;",
                            "int64_t t1 = t0 + T < N ? t0 + T : N; best_idx = -1;", "dseq"),
    "start_unmasked": ("masked[p] = 1;\n        for", "masked[p] = 0;\n        for", "dseq"),
    "pick_unmasked": ("masked[w] = 1;\n            p = w;", "p = w;", "dseq"),
    "transposed_dot": ("s += (double)ep[k] * (double)ec[k];",
                       "s += (double)ep[k] * (double)ec[(k + 1) % D];", "dseq"),
    "centroid_newest_only": ("for (int32_t i = 0; i < n_members; ++i)\n        for (int32_t k = 0; k < D; ++k) C[k]",
                             "for (int32_t i = n_members - 1; i < n_members; ++i)\n        for (int32_t k = 0; k < D; ++k) C[k]",
                             "centroid"),
    "centroid_drops_start": ("for (int32_t i = 0; i < n_members; ++i)\n        for (int32_t k = 0; k < D; ++k) C[k]",
                             "for (int32_t i = 1; i < n_members; ++i)\n        for (int32_t k = 0; k < D; ++k) C[k]",
                             "centroid"),
    "centroid_zero_reading": ("            d[c] = 1.0;\n            continue;", "            d[c] = 0.0;\n            continue;",
                              "centroid"),
    "diff_sign": ("double diff = (double)x[k] - (double)w[k];",
                  "double diff = (double)x[k] + (double)w[k];", "bmu"),
    "bmu_ties_to_highest": ("if (best_j < 0 || d < best) {",
                            "if (best_j < 0 || d <= best) {", "bmu"),
    "som_dropped_dy": ("h = exp(-(double)(dx * dx + dy * dy) / (2.0 * sigma * sigma));",
                       "h = exp(-(double)(dx * dx) / (2.0 * sigma * sigma));", "som"),
    "som_no_half": ("h = exp(-(double)(dx * dx + dy * dy) / (2.0 * sigma * sigma));",
                    "h = exp(-(double)(dx * dx + dy * dy) / (sigma * sigma));", "som"),
    "som_circular_window": ("if (h == 0.0) continue;",
                            "if (h == 0.0 || dx * dx + dy * dy > (int64_t)radius * radius) continue;",
                            "som"),
    "som_zero_unassigned": (": (double)w[k];", ": 0.0;", "som"),
    "som_transposed_grid": ("const int64_t xj = j % side_x, yj = j / side_x;",
                            "const int64_t xj = j / side_y, yj = j % side_y;", "som"),
    "som_last_sample_dropped": ("for (int64_t i = 0; i < n; ++i) {\n            const int64_t c = bmu[i];",
                                "for (int64_t i = 0; i < n - 1; ++i) {\n            const int64_t c = bmu[i];",
                                "som"),
    "bmu_dropped_term": ("for (int32_t k = 0; k < D; ++k) {\n        double diff",
                         "for (int32_t k = 1; k < D; ++k) {\n        double diff", "bmu"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_a_pin(name, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    old, new, which = MUTANTS[name]
    src = open(_SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mut = tmp_path / f"oracle_{name}.c"
    mut.write_text(src.replace(old, new))
    lib_path = str(tmp_path / f"liboracle_{name}.so")
    oracle.compile_library(str(mut), lib_path)
    lib = oracle.load(lib_path)
    fails = {"dseq": pins_dseq, "bmu": pins_bmu, "centroid": pins_centroid,
             "som": pins_som}[which](lib)
    assert fails, f"mutant {name} passed every pin"

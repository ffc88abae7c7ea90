"""Seeded synthetic inputs shaped like the two workloads of the embedding
similarity scan.  Shared by the tests (for both the oracle and the CUDA
library) and by the benchmark; it holds none of the method's arithmetic,
only the input recipes.

Recipes (numpy ``default_rng``; independent child streams from
``SeedSequence(seed).spawn``):

* ``gaussian_table``  -- i.i.d. N(0, 1) components, rows scaled to unit norm.
* ``clustered_table`` -- ``n_centres`` centres with N(0, 1) components (not
  normalised), each row = a uniformly drawn centre + N(0, sigma^2) noise per
  component, then scaled to unit norm.  Shaped like the poem-embedding table
  of the diversity issue (8,359 x 768, unit-norm, clustered); the corpus
  itself is not available, so this stands in for it.
* ``starts``          -- B distinct start rows, ``rng.choice(N, B, replace=False)``.
* ``codebook``        -- M x D components ~ U(-1, 1).
* ``bmu_samples``     -- n x D rows from ``n_centres`` centres ~ U(-1, 1)^D plus
  N(0, sigma^2) noise, uniform labels.  Stands in for the sparse MEDLINE
  articles of the BMU paper, which are not available here.

All tables are float32, C-contiguous.
"""
from __future__ import annotations

import dataclasses

import numpy as np

_CHUNK = 1 << 14  # rows generated per block (keeps float64 temporaries small)


def _streams(seed: int, k: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(k)]


def _unit_rows(a: np.ndarray) -> np.ndarray:
    a64 = a.astype(np.float64)
    nrm = np.sqrt((a64 * a64).sum(axis=1, keepdims=True))
    nrm[nrm == 0] = 1.0
    return (a64 / nrm).astype(np.float32)


def gaussian_table(N: int, D: int, seed: int = 0) -> np.ndarray:
    (rng,) = _streams(seed, 1)
    out = np.empty((N, D), np.float32)
    for r0 in range(0, N, _CHUNK):
        r1 = min(N, r0 + _CHUNK)
        out[r0:r1] = _unit_rows(rng.standard_normal((r1 - r0, D)))
    return out


def clustered_table(N: int, D: int, n_centres: int = 64, sigma: float = 0.35,
                    seed: int = 0) -> np.ndarray:
    r_centre, r_label, r_noise = _streams(seed, 3)
    centres = r_centre.standard_normal((n_centres, D))
    labels = r_label.integers(0, n_centres, size=N)
    out = np.empty((N, D), np.float32)
    for r0 in range(0, N, _CHUNK):
        r1 = min(N, r0 + _CHUNK)
        rows = centres[labels[r0:r1]] + sigma * r_noise.standard_normal((r1 - r0, D))
        out[r0:r1] = _unit_rows(rows)
    return out


def starts(N: int, B: int, seed: int = 0) -> np.ndarray:
    (rng,) = _streams(seed + 1_000_003, 1)
    return rng.choice(N, size=B, replace=False).astype(np.int32)


def codebook(M: int, D: int, seed: int = 0) -> np.ndarray:
    (rng,) = _streams(seed + 2_000_003, 1)
    out = np.empty((M, D), np.float32)
    for r0 in range(0, M, _CHUNK):
        r1 = min(M, r0 + _CHUNK)
        out[r0:r1] = rng.uniform(-1.0, 1.0, size=(r1 - r0, D))
    return out


def bmu_samples(n: int, D: int, n_centres: int = 32, sigma: float = 0.2,
                seed: int = 0) -> np.ndarray:
    r_centre, r_label, r_noise = _streams(seed + 3_000_003, 3)
    centres = r_centre.uniform(-1.0, 1.0, size=(n_centres, D))
    labels = r_label.integers(0, n_centres, size=n)
    out = np.empty((n, D), np.float32)
    for r0 in range(0, n, _CHUNK):
        r1 = min(n, r0 + _CHUNK)
        out[r0:r1] = centres[labels[r0:r1]] + sigma * r_noise.standard_normal((r1 - r0, D))
    return out


@dataclasses.dataclass(frozen=True)
class DiversityConfig:
    name: str
    N: int
    D: int
    B: int
    L: int
    kind: str  # "gaussian" | "clustered"
    oracle_seqs: int  # sequences the oracle follows under teacher forcing

    def table(self, seed: int = 0) -> np.ndarray:
        if self.kind == "gaussian":
            return gaussian_table(self.N, self.D, seed)
        return clustered_table(self.N, self.D, seed=seed)

    def starts(self, seed: int = 0) -> np.ndarray:
        return starts(self.N, self.B, seed)


@dataclasses.dataclass(frozen=True)
class BMUConfig:
    name: str
    n: int
    M: int
    D: int
    oracle_samples: int

    def samples(self, seed: int = 0) -> np.ndarray:
        return bmu_samples(self.n, self.D, seed=seed)

    def codebook(self, seed: int = 0) -> np.ndarray:
        return codebook(self.M, self.D, seed)


DIVERSITY = {
    "tiny": DiversityConfig("tiny N=512 D=64 B=8 L=32", 512, 64, 8, 32, "gaussian", 8),
    "page1": DiversityConfig("page-1 shape N=8359 D=768 B=3584 L=256", 8359, 768, 3584, 256,
                             "clustered", 64),
    "d384": DiversityConfig("dim sweep N=8359 D=384 B=3584 L=256", 8359, 384, 3584, 256,
                            "clustered", 64),
    "d1024": DiversityConfig("dim sweep N=8359 D=1024 B=3584 L=256", 8359, 1024, 3584, 256,
                             "clustered", 64),
    "scale": DiversityConfig("scale-up N=131072 D=768 B=8192 L=128", 131072, 768, 8192, 128,
                             "clustered", 64),
    # a mid-size table for profiling the Gram product and the cluster walk on
    # a few GB of device memory (G is 4.3 GB); not a benchmark configuration
    "n32k": DiversityConfig("mid-size N=32768 D=768 B=2048 L=64", 32768, 768, 2048, 64,
                            "clustered", 16),
}

BMU = {
    "som256": BMUConfig("SOM 256x256 M=65536 n=131072 D=256", 131072, 65536, 256, 4096),
    "som512": BMUConfig("SOM 512x512 M=262144 n=262144 D=256", 262144, 262144, 256, 4096),
}


# SOM epoch (BMU search, then the batch-map neighbourhood update) on the BMU
# configurations' maps.  The pages give no neighbourhood width; these take a
# mid-training Gaussian of sigma = 3 grid steps cut at radius 3 sigma.
SOM_SIDES = {"som256": (256, 256), "som512": (512, 512)}
SOM_SIGMA = 3.0
SOM_RADIUS = 9
SOM_EPOCH = {"som256_epoch": "som256", "som512_epoch": "som512"}

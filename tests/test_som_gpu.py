"""GPU parity of the SOM neighbourhood update and of whole epochs against the
CPU oracle, through the C ABI.

Tolerance: the kernels sum samples per neuron exactly (64-bit fixed point),
then smooth and divide in fp32.  Each smoothing pass is a positive-weighted sum of at most
2R + 1 terms, so the error of num / den is bounded by about
(2 (2R + 1) + 3) 2^-24 max_i |x_i|, under 2.5e-6 max|x| for R <= 9; the
tests allow 1e-5 max|x| absolute.  Epochs are checked under teacher forcing:
the search's indices are checked as in the BMU tests, and the oracle's update
then uses the GPU's indices."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads
from parity import check_bmu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 1e-5


@pytest.fixture(scope="module")
def es():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from embedding_similarity_scan_gb300 import build as esb

    esb.build()
    import embedding_similarity_scan_gb300 as mod

    mod.load()
    return mod


@pytest.fixture(autouse=True)
def _reset_options(es):
    yield
    for name, v in (("engine", 0), ("tile_n", 0), ("grid", 0), ("pair", 1)):
        es.dseq_set_option(name, v)


def _check_update(X, bmu, W_old, W_new, sx, sy, sigma, R, neurons=None):
    want = oracle.som_update(X, bmu, W_old, sx, sy, sigma, R, neurons=neurons)
    got = W_new if neurons is None else W_new[np.asarray(neurons)]
    tol = TOL * max(1.0, float(np.abs(X).max()))
    err = np.abs(got.astype(np.float64) - want)
    worst = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, f"update differs by {err.max()} (tol {tol}) at {worst}"
    return float(err.max())


def _data(n, sx, sy, D, seed, hot=False):
    rng = np.random.default_rng(seed)
    X = workloads.bmu_samples(n, D, seed=seed)
    W = workloads.codebook(sx * sy, D, seed=seed)
    if hot:  # most samples on a few neurons, as clustered data gives
        bmu = rng.choice(rng.integers(0, sx * sy, 6), size=n).astype(np.int32)
    else:
        bmu = rng.integers(0, sx * sy, n).astype(np.int32)
    return X, W, bmu


CASES = [
    # n, side_x, side_y, D, sigma, radius
    (3000, 24, 20, 40, 1.5, 4),
    (3000, 24, 20, 40, 0.0, 0),
    (5000, 33, 17, 256, 3.0, 9),
    (700, 1, 50, 37, 2.0, 5),      # one map column
    (700, 50, 1, 37, 2.0, 5),      # one map row
    (1, 3, 3, 1, 1.0, 1),
    (4000, 64, 64, 33, 0.7, 1),
    (2500, 10, 12, 300, 2.0, 3),   # D > 256: the grouped sums take two passes
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "n{}_{}x{}_D{}_s{}_R{}".format(*c))
@pytest.mark.parametrize("hot", [False, True])
def test_update_parity(es, case, hot):
    n, sx, sy, D, sigma, R = case
    X, W, bmu = _data(n, sx, sy, D, seed=n + sx, hot=hot)
    Wd = torch.from_numpy(W.copy()).cuda()
    es.som_update(torch.from_numpy(X).cuda(), torch.from_numpy(bmu).cuda(), Wd, sx, sy, sigma, R)
    torch.cuda.synchronize()
    _check_update(X, bmu, W, Wd.cpu().numpy(), sx, sy, sigma, R)


@pytest.mark.parametrize("seed", range(8))
def test_random_shapes_update(es, seed):
    """Seeded random map shapes, dimensions, sample counts, neighbourhood
    widths and radii (up to 40, beyond the usual 3 sigma), against the
    oracle."""
    rng = np.random.default_rng(3000 + seed)
    sx, sy = int(rng.integers(1, 90)), int(rng.integers(1, 90))
    D = int(rng.choice([1, 7, 32, 100, 256]))
    n = int(rng.integers(1, 4000))
    R = int(rng.integers(0, 41))
    sigma = 0.0 if R == 0 else float(rng.uniform(R / 9.0, R / 2.0 + 0.5))
    X, W, bmu = _data(n, sx, sy, D, seed=seed, hot=bool(seed % 2))
    Wd = torch.from_numpy(W).cuda()
    es.som_update(torch.from_numpy(X).cuda(), torch.from_numpy(bmu).cuda(), Wd, sx, sy, sigma, R)
    torch.cuda.synchronize()
    _check_update(X, bmu, W, Wd.cpu().numpy(), sx, sy, sigma, R)


def test_update_one_neuron_takes_every_sample(es):
    """Every sample on one neuron: its grouped samples straddle every chunk
    boundary, so all of its sums are added with atomics into a cleared row;
    a second neuron gets its own small run."""
    n, sx, sy, D, sigma, R = 5000, 16, 16, 200, 2.0, 4
    X, W, _ = _data(n, sx, sy, D, seed=77)
    bmu = np.zeros(n, np.int32)
    bmu[-7:] = 129
    Wd = torch.from_numpy(W.copy()).cuda()
    es.som_update(torch.from_numpy(X).cuda(), torch.from_numpy(bmu).cuda(), Wd, sx, sy, sigma, R)
    torch.cuda.synchronize()
    _check_update(X, bmu, W, Wd.cpu().numpy(), sx, sy, sigma, R)


def test_update_bitwise_reproducible(es):
    # the per-neuron sums are exact integers, so the order in which the
    # atomics land cannot change a bit of the result
    X, W, bmu = _data(6000, 32, 32, 96, seed=21, hot=True)
    Xd, Bd = torch.from_numpy(X).cuda(), torch.from_numpy(bmu).cuda()
    outs = []
    for _ in range(3):
        Wd = torch.from_numpy(W.copy()).cuda()
        es.som_update(Xd, Bd, Wd, 32, 32, 2.5, 7)
        outs.append(Wd.cpu().numpy())
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


@pytest.mark.parametrize("scale", [1e-30, 1e-6, 1e6, 1e30])
def test_update_value_scale(es, scale):
    # the fixed-point scale follows max |x|: parity holds at any magnitude
    X, W, bmu = _data(2000, 16, 12, 40, seed=22)
    X = (X * np.float32(scale)).astype(np.float32)
    W = (W * np.float32(scale)).astype(np.float32)
    Wd = torch.from_numpy(W.copy()).cuda()
    es.som_update(torch.from_numpy(X).cuda(), torch.from_numpy(bmu).cuda(), Wd, 16, 12, 1.3, 3)
    want = oracle.som_update(X, bmu, W, 16, 12, 1.3, 3)
    err = np.abs(Wd.cpu().numpy().astype(np.float64) - want).max()
    assert err <= TOL * float(np.abs(X).max()), f"error {err} at scale {scale}"


def test_update_host_buffers(es):
    X, W, bmu = _data(2000, 20, 16, 48, seed=4)
    Wh = W.copy()
    es.som_update(X, bmu, Wh, 20, 16, 1.2, 3)
    _check_update(X, bmu, W, Wh, 20, 16, 1.2, 3)


def test_update_untouched_neurons_keep_rows(es):
    X, W, _ = _data(100, 30, 30, 16, seed=5)
    bmu = np.full(100, 0, np.int32)  # every sample on the corner neuron
    Wd = torch.from_numpy(W.copy()).cuda()
    es.som_update(torch.from_numpy(X).cuda(), torch.from_numpy(bmu).cuda(), Wd, 30, 30, 1.0, 2)
    got = Wd.cpu().numpy()
    far = np.ones(900, bool)
    far[[r * 30 + c for r in range(3) for c in range(3)]] = False
    assert np.array_equal(got[far], W[far])
    _check_update(X, bmu, W, got, 30, 30, 1.0, 2)


def test_update_no_samples(es):
    W = workloads.codebook(12, 8, seed=1)
    Wd = torch.from_numpy(W.copy()).cuda()
    es.som_update(torch.empty((0, 8), dtype=torch.float32, device="cuda"),
                  torch.empty(0, dtype=torch.int32, device="cuda"), Wd, 4, 3, 1.0, 1)
    assert np.array_equal(Wd.cpu().numpy(), W)


def test_update_invalid(es):
    X, W, bmu = _data(50, 8, 8, 16, seed=6)
    Xd, Bd = torch.from_numpy(X).cuda(), torch.from_numpy(bmu).cuda()
    Wd = torch.from_numpy(W.copy()).cuda()
    for sigma, R in ((1.0, 10), (1.0, 256), (-1.0, 0), (float("nan"), 1)):
        with pytest.raises(es.DseqError):
            es.som_update(Xd, Bd, Wd, 8, 8, sigma, R)
    bad = Bd.clone()
    bad[7] = 64  # out of the 8 x 8 map
    with pytest.raises(es.DseqError, match="out of range"):
        es.som_update(Xd, bad, Wd, 8, 8, 1.0, 2)
    Xn = Xd.clone()
    Xn[3, 5] = float("inf")
    with pytest.raises(es.DseqError):
        es.som_update(Xn, Bd, Wd, 8, 8, 1.0, 2)
    assert np.array_equal(Wd.cpu().numpy(), W), "a failed update changed W"
    with pytest.raises(ValueError):
        es.som_update(Xd, Bd, Wd.double(), 8, 8, 1.0, 2)


@pytest.mark.parametrize("engine", ["tc_pair", "tc", "ffma"])
def test_epoch_small(es, engine):
    n, sx, sy, D = 3000, 32, 24, 64
    X = workloads.bmu_samples(n, D, seed=8)
    W = workloads.codebook(sx * sy, D, seed=8)
    es.dseq_set_option("engine", 1 if engine == "ffma" else 0)
    es.dseq_set_option("pair", 1 if engine == "tc_pair" else 0)
    Wd = torch.from_numpy(W.copy()).cuda()
    bmu, dist = es.som_epoch(torch.from_numpy(X).cuda(), Wd, sx, sy, 2.0, 6)
    torch.cuda.synchronize()
    bmu, dist = bmu.cpu().numpy(), dist.cpu().numpy()
    check_bmu(X, W, np.arange(n), bmu, dist)
    _check_update(X, bmu, W, Wd.cpu().numpy(), sx, sy, 2.0, 6)
    assert es.dseq_last_stat("update_ns") > 0


def test_epoch_host_buffers_and_repeat(es):
    n, sx, sy, D = 1500, 16, 16, 32
    X = workloads.bmu_samples(n, D, seed=9)
    W0 = workloads.codebook(sx * sy, D, seed=9)
    Wh = W0.copy()
    bmu1, dist1 = es.som_epoch(X, Wh, sx, sy, 1.5, 4)
    check_bmu(X, W0, np.arange(n), bmu1, dist1)
    _check_update(X, bmu1, W0, Wh, sx, sy, 1.5, 4)
    W1 = Wh.copy()
    bmu2, dist2 = es.som_epoch(X, Wh, sx, sy, 1.0, 3)  # a second epoch on the trained map
    check_bmu(X, W1, np.arange(n), bmu2, dist2)
    _check_update(X, bmu2, W1, Wh, sx, sy, 1.0, 3)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["som256", "som512"])
def test_epoch_full_size_sampled(es, name):
    cfg = workloads.BMU[name]
    sx, sy = workloads.SOM_SIDES[name]
    X = cfg.samples(seed=0)
    W = cfg.codebook(seed=0)
    Wd = torch.from_numpy(W.copy()).cuda()
    bmu, dist = es.som_epoch(torch.from_numpy(X).cuda(), Wd, sx, sy, workloads.SOM_SIGMA,
                             workloads.SOM_RADIUS)
    torch.cuda.synchronize()
    bmu, dist = bmu.cpu().numpy(), dist.cpu().numpy()
    rng = np.random.default_rng(1)
    sample = rng.choice(cfg.n, size=min(cfg.oracle_samples, 1024), replace=False)
    check_bmu(X, W, sample, bmu, dist)
    # neurons: random ones, the map's corners, and the most-hit neurons' rows
    hot = np.argsort(np.bincount(bmu, minlength=sx * sy))[-16:]
    neurons = np.unique(np.concatenate([rng.choice(sx * sy, 112, replace=False),
                                        [0, sx - 1, sx * (sy - 1), sx * sy - 1], hot]))
    _check_update(X, bmu, W, Wd.cpu().numpy(), sx, sy, workloads.SOM_SIGMA, workloads.SOM_RADIUS,
                  neurons=neurons)

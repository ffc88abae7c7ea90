"""GPU parity of the best-matching-unit search (both engines) against the
CPU oracle, through the C ABI; worked cases, edge cases, full sizes."""
from __future__ import annotations

import os

import numpy as np
import pytest

import workloads
from parity import check_bmu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


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
    for name, v in (("engine", 0), ("tile_n", 0), ("grid", 0), ("pair", 1), ("slice", 0),
                    ("fault_skip_copy", 0), ("timeout_ms", 10000)):
        es.dseq_set_option(name, v)


def _bmu(es, X, W, engine=0, tile_n=0, pair=1):
    es.dseq_set_option("engine", engine)
    es.dseq_set_option("tile_n", tile_n)
    es.dseq_set_option("pair", pair)
    idx, dist = es.bmu_search(torch.from_numpy(X).cuda(), torch.from_numpy(W).cuda())
    torch.cuda.synchronize()
    return idx.cpu().numpy(), dist.cpu().numpy()


SMALL = [
    (300, 1000, 40),    # ragged n, M, D
    (128, 256, 256),    # exactly one unit
    (1, 1, 1),
    (5, 3000, 7),
    (1000, 700, 300),   # D not a multiple of 32, several K blocks
    (40, 300, 16384),   # the largest D the API takes
]


@pytest.mark.parametrize("engine", ["tc_pair", "tc", "ffma"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"n{c[0]}_M{c[1]}_D{c[2]}")
def test_small(es, engine, case):
    n, M, D = case
    X = workloads.bmu_samples(n, D, seed=n + M)
    W = workloads.codebook(M, D, seed=n + M)
    idx, dist = _bmu(es, X, W, int(engine == "ffma"), pair=int(engine == "tc_pair"))
    check_bmu(X, W, np.arange(n), idx, dist)


def test_lattice_golden(es):
    W = np.array([[a, b] for a in range(-3, 4) for b in range(-3, 4)], np.float32)
    rows = [l.split() for l in open(os.path.join(GOLDEN, "bmu_lattice.txt"))
            if l.startswith("sample")]
    X = np.array([[float(r[1]), float(r[2])] for r in rows], np.float32)
    want = [int(r[3]) for r in rows]
    dwant = np.array([float(r[4]) for r in rows])
    for engine, pair in ((0, 1), (0, 0), (1, 0)):
        idx, dist = _bmu(es, X, W, engine, pair=pair)
        assert idx.tolist() == want
        assert np.allclose(dist, dwant, atol=1e-5)


def test_samples_in_codebook_and_duplicates(es):
    rng = np.random.default_rng(4)
    W = rng.uniform(-1, 1, (500, 64)).astype(np.float32)
    W[300] = W[17]
    W[499] = W[2]
    X = W[[17, 300, 2, 499, 123]].copy()
    for engine in (0, 1):
        idx, dist = _bmu(es, X, W, engine)
        assert idx.tolist() == [17, 17, 2, 2, 123]
        assert np.all(np.abs(dist) <= 1e-5 * 2 * (W[[17, 17, 2, 2, 123]] ** 2).sum(1))


def test_scale_invariance_of_split(es):
    """Rows of very different magnitudes (the per-row power-of-two scaling)."""
    rng = np.random.default_rng(8)
    W = rng.uniform(-1, 1, (700, 32)).astype(np.float32)
    W[::3] *= 1e3
    W[1::3] *= 1e-3
    X = (W[rng.integers(0, 700, 400)] + rng.normal(0, 1e-2, (400, 32))).astype(np.float32)
    idx, dist = _bmu(es, X, W)
    check_bmu(X, W, np.arange(400), idx, dist)


def test_tile_width_does_not_change_result(es):
    """Neither the neuron-chunk width nor CTA pairs reorder a dot product."""
    X = workloads.bmu_samples(2000, 96, seed=2)
    W = workloads.codebook(3000, 96, seed=2)
    ref = _bmu(es, X, W, tile_n=256, pair=0)
    for tn in (32, 128, 160):
        for pair in (0, 1):
            got = _bmu(es, X, W, tile_n=tn, pair=pair)
            assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


@pytest.mark.parametrize("D", [64, 30])
def test_unaligned_operands(es, D):
    """Operands that start 4 bytes past a 16-byte boundary: the FFMA engine
    stages them element by element, and both engines give the same result
    as for aligned copies of the same values."""
    n, M = 300, 700
    X = workloads.bmu_samples(n, D, seed=11)
    W = workloads.codebook(M, D, seed=11)

    def unaligned(A):
        buf = torch.zeros(A.size + 1, dtype=torch.float32, device="cuda")
        buf[1:].copy_(torch.from_numpy(A).reshape(-1).cuda())
        view = buf[1:].view(A.shape)
        assert view.data_ptr() % 16 == 4
        return view

    Xu, Wu = unaligned(X), unaligned(W)
    for engine in (1, 0):
        ref = _bmu(es, X, W, engine)
        es.dseq_set_option("engine", engine)
        idx, dist = es.bmu_search(Xu, Wu)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ref[0]) and np.array_equal(dist.cpu().numpy(), ref[1])
        check_bmu(X, W, np.arange(n), ref[0], ref[1])


@pytest.mark.parametrize("slice_chunks,grid", [(3, 0), (2, 8), (1, 4), (5, 2)])
def test_slices_and_segments_do_not_change_result(es, slice_chunks, grid):
    """Several codebook slices, a narrow last slice and (with few CTA pairs
    and many segments) empty segments: the same bits as one slice and as the
    single-CTA streaming kernel."""
    X = workloads.bmu_samples(700, 64, seed=12)    # 6 sample blocks (3 pairs)
    W = workloads.codebook(1700, 64, seed=12)      # 7 chunks of 256 neurons
    ref = _bmu(es, X, W, pair=0)
    check_bmu(X, W, np.arange(700), ref[0], ref[1])
    es.dseq_set_option("slice", slice_chunks)
    es.dseq_set_option("grid", grid)
    got = _bmu(es, X, W, pair=1)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


@pytest.mark.parametrize("pair,D", [(1, 64), (1, 300), (0, 64)],
                         ids=["resident", "streaming_pair", "single_cta"])
def test_pipeline_timeout_returns_cleanly(es, pair, D):
    """CTA 0 leaves out one copy of its first codebook stage: the waits on
    that stage run out after the time limit, the call returns DSEQ_ETIMEOUT,
    and the GPU stays usable (the next call gives the same bits as before)."""
    X = workloads.bmu_samples(600, D, seed=13)
    W = workloads.codebook(900, D, seed=13)
    ref = _bmu(es, X, W, pair=pair)
    es.dseq_set_option("timeout_ms", 300)
    es.dseq_set_option("fault_skip_copy", 1)
    with pytest.raises(es.DseqError) as ei:
        _bmu(es, X, W, pair=pair)
    assert ei.value.code == es.DSEQ_ETIMEOUT
    es.dseq_set_option("fault_skip_copy", 0)
    es.dseq_set_option("timeout_ms", 10000)
    got = _bmu(es, X, W, pair=pair)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


@pytest.mark.parametrize("seed", range(10))
def test_random_shapes(es, seed):
    """Seeded random sample counts, codebook sizes, dimensions (both sides of
    the resident-sample limit), chunk widths and pair modes, against the
    oracle."""
    rng = np.random.default_rng(2000 + seed)
    n = int(rng.integers(1, 1500))
    M = int(rng.integers(1, 3000))
    D = int(rng.choice([1, 5, 32, 100, 256, 300, 513]))
    tile_n = int(rng.choice([0, 32, 96, 256]))
    pair = int(rng.integers(0, 2))
    X = workloads.bmu_samples(n, D, seed=seed)
    W = workloads.codebook(M, D, seed=seed)
    idx, dist = _bmu(es, X, W, 0, tile_n=tile_n, pair=pair)
    check_bmu(X, W, np.arange(n), idx, dist)


def test_host_buffers(es):
    X = workloads.bmu_samples(257, 24, seed=6)
    W = workloads.codebook(513, 24, seed=6)
    idx, dist = es.bmu_search(X, W)
    assert isinstance(idx, np.ndarray)
    check_bmu(X, W, np.arange(257), idx, dist)


def test_invalid(es):
    X = np.zeros((4, 8), np.float32)
    W = np.ones((6, 8), np.float32)
    W[2, 2] = np.inf
    with pytest.raises(es.DseqError) as ei:
        es.bmu_search(torch.from_numpy(X).cuda(), torch.from_numpy(W).cuda())
    assert ei.value.code == es.DSEQ_ENONFINITE
    with pytest.raises(ValueError):
        es.bmu_search(X, np.ones((6, 9), np.float32))


@pytest.mark.parametrize("name,engine", [("som256", 0), ("som512", 0), ("som256", 1)],
                         ids=lambda c: str(c))
def test_full_size_sampled(es, name, engine):
    """The full configurations (and som256 on the FFMA engine), checked on a
    seeded sample of rows."""
    cfg = workloads.BMU[name]
    X = cfg.samples(seed=0)
    W = cfg.codebook(seed=0)
    idx, dist = _bmu(es, X, W, engine)
    sample = np.sort(np.random.default_rng(0).choice(cfg.n, cfg.oracle_samples, replace=False))
    counts = check_bmu(X, W, sample, idx, dist)
    # how much the near-tie reading matters at this size: samples in each band
    print(f"\n{name} engine {engine}: {counts}")
    assert np.all((idx >= 0) & (idx < cfg.M)) and np.all(dist >= 0)

"""GPU parity of the diversity scan (both engines) against the CPU oracle,
through the C ABI, under teacher forcing; edge cases and error paths."""
from __future__ import annotations

import numpy as np
import pytest

import workloads
from parity import check_centroid_teacher_forced, check_dseq_teacher_forced, check_picks_valid

pytestmark = pytest.mark.gpu

DEFAULT_PAIR = 1

torch = pytest.importorskip("torch")


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
    for name, v in (("engine", 0), ("tile_n", 0), ("tile_n2", 0), ("grid", 0), ("timeout_ms", 10000),
                    ("fault_skip_arrive", 0), ("pair", DEFAULT_PAIR), ("storage", 0),
                    ("criterion", 0), ("resume", 0), ("compact", 1), ("isolate_epilogue", 0),
                    ("gram", 2), ("walk", 0)):
        es.dseq_set_option(name, v)


def _run(es, E, starts, L, mask=None, trace_seqs=None, engine=0, tile_n=0, grid=0,
         pair=None, storage=0, criterion=0, tile_n2=0, gram=0):
    """One context, one run.  gram = 0 (default here) keeps the tests that
    target the per-iteration kernels on them; gram = 1 runs the Gram engine,
    2 lets the library choose."""
    dev = torch.device("cuda")
    es.dseq_set_option("gram", gram)
    es.dseq_set_option("engine", engine)
    es.dseq_set_option("tile_n", tile_n)
    es.dseq_set_option("tile_n2", tile_n2)
    es.dseq_set_option("grid", grid)
    es.dseq_set_option("pair", DEFAULT_PAIR if pair is None else pair)
    es.dseq_set_option("storage", storage)
    es.dseq_set_option("criterion", criterion)
    ctx = es.dseq_create(torch.from_numpy(E).to(dev))
    try:
        st = torch.from_numpy(np.asarray(starts, np.int32)).to(dev)
        mk = None if mask is None else torch.from_numpy(np.asarray(mask, np.uint8)).to(dev)
        if trace_seqs is None:
            picks = es.dseq_run(ctx, st, L, mask=mk)
            torch.cuda.synchronize()
            return picks.cpu().numpy(), None
        tr = torch.from_numpy(np.asarray(trace_seqs, np.int32)).to(dev)
        picks, trace = es.dseq_run_trace(ctx, st, L, tr, mask=mk)
        torch.cuda.synchronize()
        return picks.cpu().numpy(), trace.cpu().numpy()
    finally:
        ctx.close()


SMALL = [
    # (N, D, B, L, kind, masked fraction)
    (512, 64, 8, 32, "gaussian", 0.0),      # the tiny configuration
    (1000, 96, 200, 16, "clustered", 0.0),  # ragged N, B, several tiles
    (777, 33, 130, 20, "gaussian", 0.05),   # D not a multiple of 32, masked rows
    (300, 1, 5, 10, "gaussian", 0.0),       # D = 1: every distance is 0 or 2
    (2049, 200, 129, 12, "clustered", 0.1),
]


@pytest.mark.parametrize("engine", ["tc", "tc_pair", "ffma"])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_small_teacher_forced(es, engine, case):
    N, D, B, L, kind, frac = case
    E = workloads.gaussian_table(N, D, seed=N) if kind == "gaussian" else \
        workloads.clustered_table(N, D, n_centres=16, seed=N)
    starts = workloads.starts(N, B, seed=N)
    mask = None
    if frac > 0:
        rng = np.random.default_rng(N)
        mask = (rng.random(N) < frac).astype(np.uint8)
        mask[starts[: B // 3]] = 1  # some starts are masked themselves
    trace_seqs = np.arange(B, dtype=np.int32) if B <= 200 else \
        np.sort(np.random.default_rng(1).choice(B, 64, replace=False)).astype(np.int32)
    picks, trace = _run(es, E, starts, L, mask, trace_seqs, engine=int(engine == "ffma"),
                        pair=int(engine == "tc_pair"))
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, trace_seqs)


EXTREME = [
    # (N, D, B, L): the largest D the API takes, a table narrower than one
    # chunk run to its full ordering, one sequence, a wide D with many blocks
    (300, 16384, 16, 4),
    (20, 8, 3, 19),
    (1500, 64, 1, 40),
    (700, 4096, 520, 6),
]


@pytest.mark.parametrize("engine", ["tc", "tc_pair", "ffma"])
@pytest.mark.parametrize("case", EXTREME, ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_extreme_shapes_teacher_forced(es, engine, case):
    N, D, B, L = case
    E = workloads.gaussian_table(N, D, seed=D + N)
    starts = workloads.starts(N, B, seed=D + N)
    tr = np.unique(np.array([0, B // 2, B - 1], np.int32))
    picks, trace = _run(es, E, starts, L, None, tr, engine=1 if engine == "ffma" else 0,
                        pair=1 if engine == "tc_pair" else 0)
    check_picks_valid(starts, None, picks, N)
    check_dseq_teacher_forced(E, starts, None, picks, trace, tr)


def test_picks_identical_across_candidate_tiles(es):
    """Candidate tiling does not reorder any dot product, so the picks (and
    the running minima) must be bit-identical for every tile width."""
    N, D, B, L = 3000, 128, 300, 24
    E = workloads.clustered_table(N, D, n_centres=8, seed=11)
    starts = workloads.starts(N, B, seed=11)
    ref, ref_tr = _run(es, E, starts, L, trace_seqs=[0, 7, 299], tile_n=256, pair=0)
    for tn in (32, 96, 128, 224):
        got, tr = _run(es, E, starts, L, trace_seqs=[0, 7, 299], tile_n=tn, pair=0)
        assert np.array_equal(got, ref), f"tile_n={tn} changes the picks"
        assert np.array_equal(tr, ref_tr), f"tile_n={tn} changes the running minima"
    got, _ = _run(es, E, starts, L, grid=7, pair=0)
    assert np.array_equal(got, ref), "grid size changes the picks"
    # CTA pairs run the same K order into the same fp32 accumulators
    for tn in (64, 224, 256):
        got, tr = _run(es, E, starts, L, trace_seqs=[0, 7, 299], tile_n=tn, pair=1)
        assert np.array_equal(got, ref), f"pair mode, tile_n={tn} changes the picks"
        assert np.array_equal(tr, ref_tr), f"pair mode, tile_n={tn} changes the running minima"
    got, _ = _run(es, E, starts, L, grid=6, pair=1)
    assert np.array_equal(got, ref), "pair mode with 3 clusters changes the picks"
    # two chunk widths (wide chunks, then narrow ones)
    for tn, tn2, pair in ((256, 192, 1), (256, 64, 1), (224, 32, 0), (128, 96, 0)):
        got, tr = _run(es, E, starts, L, trace_seqs=[0, 7, 299], tile_n=tn, tile_n2=tn2,
                       pair=pair)
        assert es.dseq_last_stat("tile_n2") == tn2 or es.dseq_last_stat("n_wide") > 0
        assert np.array_equal(got, ref), f"widths {tn}/{tn2} (pair {pair}) change the picks"
        assert np.array_equal(tr, ref_tr), f"widths {tn}/{tn2} change the running minima"


@pytest.mark.parametrize("pair", [1, 0])
def test_mixed_widths_teacher_forced(es, pair):
    """The default plan at a page-1-like width mix, against the oracle, with a
    mask and a ragged last chunk."""
    N, D, B, L = 2085, 96, 700, 20
    E = workloads.clustered_table(N, D, n_centres=12, seed=5)
    starts = workloads.starts(N, B, seed=5)
    mask = (np.random.default_rng(5).random(N) < 0.1).astype(np.uint8)
    mask[starts] = 0
    tr = np.array([0, 1, 255, 256, 699], np.int32)
    picks, trace = _run(es, E, starts, L, mask, tr, tile_n=256, tile_n2=96, pair=pair)
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, tr)


def test_exhaustion_boundary(es):
    """L = every candidate a sequence has left: the last picks are forced."""
    N, D = 97, 16
    E = workloads.gaussian_table(N, D, seed=3)
    mask = np.zeros(N, np.uint8)
    mask[[3, 50, 96]] = 1
    starts = np.array([0, 50, 96, 10], np.int32)  # two masked starts
    L = N - 3 - 1  # sequences whose start is unmasked have N - 4 left
    with pytest.raises(es.DseqError) as ei:
        _run(es, E, starts, L + 1, mask)
    assert ei.value.code == es.DSEQ_EINVAL
    picks, trace = _run(es, E, starts, L, mask, trace_seqs=[0, 1, 2, 3])
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, [0, 1, 2, 3])


def test_orthonormal_ties_lowest_index(es):
    """Every distance between distinct rows of the identity is exactly 1, so
    every pick is a tie and the picks are the ascending unmasked indices."""
    N = 64
    E = np.eye(N, dtype=np.float32)
    starts = np.array([0, 5, 63], np.int32)
    for engine in (0, 1):
        picks, _ = _run(es, E, starts, N - 1, engine=engine)
        for b, s in enumerate(starts):
            assert picks[b].tolist() == [c for c in range(N) if c != s]


def test_square4_worked_example(es):
    E = np.array([[1, 0], [0, 1], [-1, 0], [0, -1]], np.float32) * \
        np.array([[2.0], [0.5], [3.0], [7.0]], np.float32)
    for engine in (0, 1):
        picks, _ = _run(es, E, np.array([0, 3, 1], np.int32), 3, engine=engine)
        assert picks.tolist() == [[2, 1, 3], [1, 0, 2], [3, 0, 2]]


def test_single_candidate_and_zero_length(es):
    E = workloads.gaussian_table(1, 8, seed=0)
    picks, _ = _run(es, E, np.array([0], np.int32), 0)
    assert picks.shape == (1, 0)
    E = workloads.gaussian_table(2, 8, seed=0)
    picks, _ = _run(es, E, np.array([1], np.int32), 1)
    assert picks.tolist() == [[0]]


def test_invalid_arguments(es):
    N = 50
    E = workloads.gaussian_table(N, 8, seed=0)
    for bad_starts in ([0, 50], [-1], [3, 3]):
        with pytest.raises(es.DseqError) as ei:
            _run(es, E, np.array(bad_starts, np.int32), 2)
        assert ei.value.code == es.DSEQ_EINVAL
    with pytest.raises(es.DseqError) as ei:
        _run(es, E, np.array([0], np.int32), N)
    assert ei.value.code == es.DSEQ_EINVAL
    bad = E.copy()
    bad[7, 3] = np.nan
    with pytest.raises(es.DseqError) as ei:
        es.dseq_create(torch.from_numpy(bad).cuda())
    assert ei.value.code == es.DSEQ_ENONFINITE
    bad = E.copy()
    bad[9] = 0.0
    with pytest.raises(es.DseqError) as ei:
        es.dseq_create(torch.from_numpy(bad).cuda())
    assert ei.value.code == es.DSEQ_ENONFINITE


def test_host_buffers(es):
    """Host (numpy) table, starts and picks: the library stages the copies."""
    N, D, B, L = 600, 48, 20, 10
    E = workloads.gaussian_table(N, D, seed=21)
    starts = workloads.starts(N, B, seed=21)
    ctx = es.dseq_create(E)
    try:
        host_picks = es.dseq_run(ctx, starts, L)
    finally:
        ctx.close()
    assert isinstance(host_picks, np.ndarray)
    dev_picks, _ = _run(es, E, starts, L)
    assert np.array_equal(host_picks, dev_picks)


@pytest.mark.parametrize("criterion,pair", [(0, 1), (0, 0), (1, 1)])
def test_barrier_timeout_returns_cleanly(es, criterion, pair):
    """One CTA skips its first arrival on the cross-CTA "half done" counter:
    every wait runs out after the time limit, the call returns DSEQ_ETIMEOUT,
    and the GPU stays usable (max-min pair and single CTA, centroid)."""
    N, D, B, L = 2000, 64, 512, 4
    E = workloads.gaussian_table(N, D, seed=5)
    starts = workloads.starts(N, B, seed=5)
    ref, _ = _run(es, E, starts, L, criterion=criterion, pair=pair)
    es.dseq_set_option("timeout_ms", 500)
    es.dseq_set_option("fault_skip_arrive", 1)
    with pytest.raises(es.DseqError) as ei:
        _run(es, E, starts, L, criterion=criterion, pair=pair)
    assert ei.value.code == es.DSEQ_ETIMEOUT
    es.dseq_set_option("fault_skip_arrive", 0)
    es.dseq_set_option("timeout_ms", 10000)
    again, _ = _run(es, E, starts, L, criterion=criterion, pair=pair)
    assert np.array_equal(again, ref)


@pytest.mark.parametrize("pair,criterion,storage", [(1, 0, 0), (0, 0, 0), (1, 1, 0), (1, 0, 1)])
def test_oversized_grid_returns_elaunch(es, pair, criterion, storage):
    """A "grid" option beyond the CTAs that can be co-resident: the runtime
    refuses the cooperative launch, the call returns DSEQ_ELAUNCH with the
    refusal's message and launches nothing in another form, and the next call
    with the default grid (sized from the launched variant's own occupancy)
    gives the same picks as before."""
    N, D, B, L = 20000, 64, 1024, 2
    E = workloads.gaussian_table(N, D, seed=8)
    starts = workloads.starts(N, B, seed=8)
    # 32-wide chunks: 625 chunks x 8 sequence blocks, more units than the grid
    kw = dict(pair=pair, criterion=criterion, storage=storage, tile_n=32)
    ref, _ = _run(es, E, starts, L, **kw)
    grid = es.dseq_last_stat("grid")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 0 < grid <= sms and (grid % 2 == 0 or not pair)
    with pytest.raises(es.DseqError) as ei:
        _run(es, E, starts, L, grid=1000, **kw)
    assert ei.value.code == es.DSEQ_ELAUNCH
    assert "refused" in str(ei.value)
    again, _ = _run(es, E, starts, L, grid=0, **kw)
    assert np.array_equal(again, ref)


@pytest.mark.parametrize("pair,storage", [(1, 0), (0, 0), (1, 1), (0, 1)])
def test_isolated_epilogue_runs_epilogue_and_commit(es, pair, storage):
    """The epilogue-isolated kernel (contraction compiled out, a distance that
    falls every iteration and is equal for every candidate) still folds,
    reduces and commits: every candidate ties each iteration, so every
    sequence picks the lowest candidates in order, skipping its start and the
    masked rows.  Results of the real kernel are unaffected afterwards."""
    N, D, B, L = 3000, 64, 300, 12
    E = workloads.gaussian_table(N, D, seed=12)
    starts = workloads.starts(N, B, seed=12)
    mask = np.zeros(N, np.uint8)
    mask[[1, 4, 9]] = 1
    ref, _ = _run(es, E, starts, L, mask, pair=pair, storage=storage)
    es.dseq_set_option("isolate_epilogue", 1)
    got, _ = _run(es, E, starts, L, mask, pair=pair, storage=storage)
    es.dseq_set_option("isolate_epilogue", 0)
    for b in range(B):
        want = [c for c in range(N) if not mask[c] and c != starts[b]][:L]
        assert got[b].tolist() == want, f"sequence {b}"
    again, _ = _run(es, E, starts, L, mask, pair=pair, storage=storage)
    assert np.array_equal(again, ref)


FULL = ["page1", "d384", "d1024", "scale"]


@pytest.mark.parametrize("name,engine", [(n, 0) for n in FULL] + [("page1", 1)],
                         ids=lambda c: str(c))
def test_full_size_teacher_forced(es, name, engine):
    """The full configurations, in the launch configuration the benchmark
    times (and the page-1 shape on the FFMA engine), with a seeded subset of
    sequences followed by the oracle."""
    cfg = workloads.DIVERSITY[name]
    E = cfg.table(seed=0)
    starts = cfg.starts(seed=0)
    tr = np.sort(np.random.default_rng(0).choice(cfg.B, cfg.oracle_seqs, replace=False))
    picks, trace = _run(es, E, starts, cfg.L, trace_seqs=tr.astype(np.int32), engine=engine)
    check_dseq_teacher_forced(E, starts[tr], None, picks[tr], trace, np.arange(tr.size))
    # picks of every sequence: in range, distinct, never the start
    assert np.all((picks >= 0) & (picks < cfg.N))
    srt = np.sort(picks, axis=1)
    assert not np.any(srt[:, 1:] == srt[:, :-1]), "a sequence repeats a pick"
    assert not np.any(picks == starts[:, None]), "a sequence picks its start"


# --------------------------------------------------------------------------
# fp16 table storage (fp16 in memory, fp32 arithmetic): on tables whose values are
# already fp16 numbers the stored rows equal the input up to a power-of-two
# scale, so the distances match the oracle's exact cosine distances to fp32
# accumulation error, and the same teacher-forced tolerance applies.


def _fp16_table(E):
    return E.astype(np.float16).astype(np.float32)


@pytest.mark.parametrize("pair", [1, 0])
@pytest.mark.parametrize("case", SMALL[:3] + SMALL[4:], ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_fp16_storage_teacher_forced(es, pair, case):
    N, D, B, L, kind, frac = case
    E = workloads.gaussian_table(N, D, seed=N) if kind == "gaussian" else \
        workloads.clustered_table(N, D, n_centres=16, seed=N)
    E = _fp16_table(E)
    starts = workloads.starts(N, B, seed=N)
    mask = None
    if frac > 0:
        rng = np.random.default_rng(N)
        mask = (rng.random(N) < frac).astype(np.uint8)
    trace_seqs = np.arange(min(B, 200), dtype=np.int32)
    picks, trace = _run(es, E, starts, L, mask, trace_seqs, pair=pair, storage=1)
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, trace_seqs)


def test_fp16_storage_full_size_and_agreement(es):
    """Page-1 shape with fp16 storage: teacher-forced parity on the fp16
    version of the table; on the original table, the share of picks equal to
    the fp32-accurate path is reported (the issue expects the ordering to
    survive FP16 storage)."""
    cfg = workloads.DIVERSITY["page1"]
    E = cfg.table(seed=0)
    starts = cfg.starts(seed=0)
    tr = np.sort(np.random.default_rng(0).choice(cfg.B, 32, replace=False)).astype(np.int32)
    E16 = _fp16_table(E)
    picks, trace = _run(es, E16, starts, cfg.L, trace_seqs=tr, storage=1)
    check_dseq_teacher_forced(E16, starts[tr], None, picks[tr], trace, np.arange(tr.size))
    ref, _ = _run(es, E, starts[:512], cfg.L, storage=0)
    got, _ = _run(es, E, starts[:512], cfg.L, storage=1)
    check_picks_valid(starts[:512], None, got, cfg.N)
    same_seq = float(np.mean(np.all(ref == got, axis=1)))
    same_pick = float(np.mean(ref == got))
    print(f"fp16 storage vs split: identical sequences {same_seq:.3f}, identical picks {same_pick:.3f}")


# --------------------------------------------------------------------------
# centroid criterion (the distance-from-the-centroid reading of "Issue 9-014:
# Tile Diversity Shader Inner Loop For L2 Cache Locality", section FP16
# storage (compounding optimization))


@pytest.mark.parametrize("pair", [1, 0])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_centroid_teacher_forced(es, pair, case):
    N, D, B, L, kind, frac = case
    E = workloads.gaussian_table(N, D, seed=N) if kind == "gaussian" else \
        workloads.clustered_table(N, D, n_centres=16, seed=N)
    starts = workloads.starts(N, B, seed=N)
    mask = None
    if frac > 0:
        rng = np.random.default_rng(N)
        mask = (rng.random(N) < frac).astype(np.uint8)
        mask[starts[: B // 3]] = 1
    trace_seqs = np.arange(min(B, 64), dtype=np.int32)
    picks, trace = _run(es, E, starts, L, mask, trace_seqs, pair=pair, criterion=1)
    check_picks_valid(starts, mask, picks, N)
    check_centroid_teacher_forced(E, starts, mask, picks, trace, trace_seqs)


def test_centroid_worked_example(es):
    """Four rows on which the two criteria disagree (hand-derived)."""
    c, s = np.float32(np.cos(np.radians(10.0))), np.float32(np.sin(np.radians(10.0)))
    E = np.array([[1, 0], [c, s], [-1, 0], [0, 1]], np.float32)
    for pair in (1, 0):
        got, _ = _run(es, E, np.array([0], np.int32), 3, pair=pair, criterion=1)
        assert got.tolist() == [[2, 1, 3]]
        got, _ = _run(es, E, np.array([0], np.int32), 3, pair=pair, criterion=0)
        assert got.tolist() == [[2, 3, 1]]


def test_centroid_full_size(es):
    cfg = workloads.DIVERSITY["page1"]
    E = cfg.table(seed=0)
    starts = cfg.starts(seed=0)
    tr = np.sort(np.random.default_rng(2).choice(cfg.B, 16, replace=False)).astype(np.int32)
    picks, trace = _run(es, E, starts, cfg.L, trace_seqs=tr, criterion=1)
    check_centroid_teacher_forced(E, starts[tr], None, picks[tr], trace, np.arange(tr.size))
    srt = np.sort(picks, axis=1)
    assert not np.any(srt[:, 1:] == srt[:, :-1]) and not np.any(picks == starts[:, None])


# fp16 storage on the Gram engine: G holds the inner products of the stored
# fp16 rows' unit vectors; on tables of fp16 numbers those are the oracle's
# exact cosine distances


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_gram_fp16_storage_teacher_forced(es, case):
    N, D, B, L, kind, frac = case
    E = workloads.gaussian_table(N, D, seed=N) if kind == "gaussian" else \
        workloads.clustered_table(N, D, n_centres=16, seed=N)
    E = _fp16_table(E)
    starts = workloads.starts(N, B, seed=N)
    mask = None
    if frac > 0:
        rng = np.random.default_rng(N)
        mask = (rng.random(N) < frac).astype(np.uint8)
        mask[starts[: B // 3]] = 1
    trace_seqs = np.arange(min(B, 64), dtype=np.int32)
    picks, trace = _run(es, E, starts, L, mask, trace_seqs, storage=1, gram=1)
    assert es.dseq_last_stat("gram") == 1
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, trace_seqs)


def test_gram_fp16_storage_cluster_walk(es):
    """fp16 storage on a table whose running minima need a cluster of CTAs
    (N = 30011), and in global memory: the oracle's distances on the fp16
    table, identical picks in both places."""
    N, D, B, L = 30011, 48, 9, 8
    E = _fp16_table(workloads.clustered_table(N, D, n_centres=20, seed=41))
    starts = workloads.starts(N, B, seed=41)
    tr = np.arange(B, dtype=np.int32)
    es.dseq_set_option("walk", 0)
    picks, trace = _run(es, E, starts, L, None, tr, storage=1, gram=1)
    assert es.dseq_last_stat("gram") == 1 and es.dseq_last_stat("walk") == 2
    check_dseq_teacher_forced(E, starts, None, picks, trace, tr)
    es.dseq_set_option("walk", 3)
    picks3, trace3 = _run(es, E, starts, L, None, tr, storage=1, gram=1)
    es.dseq_set_option("walk", 0)
    assert np.array_equal(picks3, picks) and np.array_equal(trace3, trace)


def test_gram_fp16_storage_full_size(es):
    """Page 1 with fp16 storage on the engine the library picks (the Gram
    engine): teacher-forced parity on the fp16 version of the table, and
    the picks against the scan's fp16-storage run (same distances up to
    fp32 rounding: near-ties aside, the same sequences)."""
    cfg = workloads.DIVERSITY["page1"]
    E16 = _fp16_table(cfg.table(seed=0))
    starts = cfg.starts(seed=0)
    tr = np.sort(np.random.default_rng(6).choice(cfg.B, 16, replace=False)).astype(np.int32)
    picks, trace = _run(es, E16, starts, cfg.L, trace_seqs=tr, storage=1, gram=2)
    assert es.dseq_last_stat("gram") == 1
    check_dseq_teacher_forced(E16, starts[tr], None, picks[tr], trace, np.arange(tr.size))
    check_picks_valid(starts, None, picks, cfg.N)
    scan, _ = _run(es, E16, starts[:256], cfg.L, storage=1, gram=0)
    same = float(np.mean(np.all(scan == picks[:256], axis=1)))
    first = float(np.mean(scan[:, 0] == picks[:256, 0]))
    print(f"fp16 storage, Gram engine vs scan: identical sequences {same:.3f}, "
          f"identical first picks {first:.3f}")
    assert first >= 0.95


def test_centroid_rejects_ffma(es):
    E = workloads.gaussian_table(100, 16, seed=1)
    with pytest.raises(es.DseqError):
        _run(es, E, np.array([0], np.int32), 3, engine=1, criterion=1)


# the centroid criterion on fp16 table storage ("Issue 9-014: Tile Diversity
# Shader Inner Loop For L2 Cache Locality", section FP16 storage (compounding
# optimization), ranks candidates by their distance from the centroid): the
# table is held as fp16 rows, the
# centroid query keeps fp32-level precision, so on tables of fp16 numbers the
# distances are the oracle's exact cosine distances to the centroid.


@pytest.mark.parametrize("pair", [1, 0])
@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_centroid_fp16_storage_teacher_forced(es, pair, case):
    N, D, B, L, kind, frac = case
    E = workloads.gaussian_table(N, D, seed=N) if kind == "gaussian" else \
        workloads.clustered_table(N, D, n_centres=16, seed=N)
    E = _fp16_table(E)
    starts = workloads.starts(N, B, seed=N)
    mask = None
    if frac > 0:
        rng = np.random.default_rng(N)
        mask = (rng.random(N) < frac).astype(np.uint8)
        mask[starts[: B // 3]] = 1
    trace_seqs = np.arange(min(B, 64), dtype=np.int32)
    picks, trace = _run(es, E, starts, L, mask, trace_seqs, pair=pair, storage=1, criterion=1)
    check_picks_valid(starts, mask, picks, N)
    check_centroid_teacher_forced(E, starts, mask, picks, trace, trace_seqs)


def test_centroid_fp16_storage_full_size_and_agreement(es):
    """Page-1 shape, centroid criterion on fp16 storage: teacher-forced
    parity on the fp16 version of the table; on the original table, the
    share of picks equal to the split-storage centroid run is reported."""
    cfg = workloads.DIVERSITY["page1"]
    E = cfg.table(seed=0)
    starts = cfg.starts(seed=0)
    tr = np.sort(np.random.default_rng(5).choice(cfg.B, 16, replace=False)).astype(np.int32)
    E16 = _fp16_table(E)
    picks, trace = _run(es, E16, starts, cfg.L, trace_seqs=tr, storage=1, criterion=1)
    check_centroid_teacher_forced(E16, starts[tr], None, picks[tr], trace, np.arange(tr.size))
    check_picks_valid(starts, None, picks, cfg.N)
    ref, _ = _run(es, E, starts[:512], cfg.L, storage=0, criterion=1)
    got, _ = _run(es, E, starts[:512], cfg.L, storage=1, criterion=1)
    check_picks_valid(starts[:512], None, got, cfg.N)
    same_seq = float(np.mean(np.all(ref == got, axis=1)))
    same_pick = float(np.mean(ref == got))
    print(f"centroid, fp16 storage vs split: identical sequences {same_seq:.3f}, "
          f"identical picks {same_pick:.3f}")


# --------------------------------------------------------------------------
# long orderings in chunks ("resume"): the driver of "Issue 9-014: Tile
# Diversity Shader Inner Loop For L2 Cache Locality" (Current Behavior) runs
# the sequences in chunks of iterations; continuing from the state left on the device must
# give exactly the picks of one long call.


@pytest.mark.parametrize("engine,pair,criterion,storage,gram,walk",
                         [(0, 1, 0, 0, 0, 0), (0, 0, 0, 0, 0, 0), (1, 0, 0, 0, 0, 0),
                          (0, 1, 1, 0, 0, 0), (0, 1, 0, 1, 0, 0), (0, 1, 1, 1, 0, 0),
                          (0, 1, 0, 0, 1, 1), (0, 1, 0, 0, 1, 2), (0, 1, 0, 0, 1, 3),
                          (0, 1, 0, 1, 1, 0)])
def test_resume_in_chunks_equals_one_call(es, engine, pair, criterion, storage, gram, walk):
    N, D, B = 300, 40, 9
    E = workloads.clustered_table(N, D, n_centres=6, seed=12)
    starts = workloads.starts(N, B, seed=12)
    mask = np.zeros(N, np.uint8)
    mask[::17] = 1
    mask[starts] = 0
    L_total = N - int(mask.sum()) - 1  # the full ordering of every sequence
    traced = np.array([0, B - 1], np.int32)
    if storage:  # fp16 storage: a table of fp16 numbers keeps the oracle exact
        E = E.astype(np.float16).astype(np.float32)
    es.dseq_set_option("engine", engine)
    es.dseq_set_option("pair", pair)
    es.dseq_set_option("criterion", criterion)
    es.dseq_set_option("storage", storage)
    es.dseq_set_option("gram", gram)
    es.dseq_set_option("walk", walk)
    ctx = es.dseq_create(torch.from_numpy(E).cuda())
    try:
        st = torch.from_numpy(starts).cuda()
        mk = torch.from_numpy(mask).cuda()
        es.dseq_set_option("resume", 0, ctx)
        whole = es.dseq_run(ctx, st, L_total, mask=mk).cpu().numpy()
        parts, traces = [], []
        for i, chunk in enumerate((50, 1, 100, L_total - 151)):
            es.dseq_set_option("resume", 0 if i == 0 else 1, ctx)
            pk, tr = es.dseq_run_trace(ctx, st, chunk, torch.from_numpy(traced).cuda(), mask=mk)
            parts.append(pk.cpu().numpy())
            traces.append(tr.cpu().numpy())
        with pytest.raises(es.DseqError):  # nothing left to pick
            es.dseq_run(ctx, st, 1, mask=mk)
        with pytest.raises(es.DseqError):  # different starts
            es.dseq_run(ctx, torch.flip(st, [0]), 1, mask=mk)
        with pytest.raises(es.DseqError):  # different mask
            es.dseq_run(ctx, st, 1)
    finally:
        ctx.close()
    chunked = np.concatenate(parts, axis=1)
    assert np.array_equal(chunked, whole)
    check_picks_valid(starts, mask, whole, N)
    # the chunks' traces, joined, follow the oracle from the starts on
    trace = np.concatenate(traces, axis=1)
    check = check_centroid_teacher_forced if criterion else check_dseq_teacher_forced
    check(E, starts, mask, chunked, trace, traced)


@pytest.mark.parametrize("pair,storage,criterion",
                         [(1, 0, 0), (0, 0, 0), (1, 1, 0), (1, 0, 1), (0, 1, 1)],
                         ids=["pair", "single", "fp16", "centroid", "fp16-centroid"])
def test_global_mask_compaction_identical(es, pair, storage, criterion):
    """A global mask that removes about a third of the table: the kernel
    scans only the unmasked rows, with the same picks and the same running
    minima (masked rows -inf in the trace) as the full scan, in one call or
    resumed in chunks; and it follows the oracle."""
    N, D, B, L = 1500, 64, 150, 24
    E = workloads.clustered_table(N, D, n_centres=12, seed=21)
    if storage:
        E = _fp16_table(E)
    starts = workloads.starts(N, B, seed=21)
    rng = np.random.default_rng(21)
    mask = (rng.random(N) < 0.33).astype(np.uint8)
    mask[starts[: B // 4]] = 1  # some starts are masked themselves
    tr = np.array([0, 7, B // 4, B - 1], np.int32)
    got = {}
    for compact in (0, 1):
        es.dseq_set_option("compact", compact)
        got[compact] = _run(es, E, starts, L, mask, tr, pair=pair, storage=storage,
                            criterion=criterion)
    assert np.array_equal(got[0][0], got[1][0])
    assert np.array_equal(got[0][1], got[1][1])
    picks, trace = got[1]
    check_picks_valid(starts, mask, picks, N)
    check = check_centroid_teacher_forced if criterion else check_dseq_teacher_forced
    check(E, starts, mask, picks, trace, tr)
    # the compacted run resumed in two chunks gives the same picks
    es.dseq_set_option("gram", 0)
    es.dseq_set_option("compact", 1)
    es.dseq_set_option("pair", pair)
    es.dseq_set_option("storage", storage)
    es.dseq_set_option("criterion", criterion)
    ctx = es.dseq_create(torch.from_numpy(E).cuda())
    try:
        st = torch.from_numpy(starts).cuda()
        mk = torch.from_numpy(mask).cuda()
        first = es.dseq_run(ctx, st, 10, mask=mk).cpu().numpy()
        es.dseq_set_option("resume", 1, ctx)
        rest = es.dseq_run(ctx, st, L - 10, mask=mk).cpu().numpy()
        es.dseq_set_option("compact", 0, ctx)
        with pytest.raises(es.DseqError):  # a different scan layout cannot resume
            es.dseq_run(ctx, st, 1, mask=mk)
    finally:
        ctx.close()
    assert np.array_equal(np.concatenate([first, rest], axis=1), picks)


def _random_case(seed):
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(2, 3000))
    D = int(rng.choice([1, 3, 17, 32, 64, 100, 257, 768]))
    B = int(rng.integers(1, min(N, 300) + 1))
    frac = float(rng.choice([0.0, 0.02, 0.1, 0.4]))
    mask = (rng.random(N) < frac).astype(np.uint8) if frac > 0 else None
    starts = rng.choice(N, B, replace=False).astype(np.int32)
    n_masked = 0 if mask is None else int(mask.sum())
    L = int(rng.integers(1, max(2, min(N - n_masked - 1, 40) + 1))) if N - n_masked - 1 >= 1 else 0
    return N, D, B, L, mask, starts


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("pair", [1, 0])
def test_random_shapes_teacher_forced(es, seed, pair):
    """Seeded random shapes, masks (dense enough to be compacted or not),
    sequence counts and lengths, against the oracle."""
    N, D, B, L, mask, starts = _random_case(seed)
    if L == 0:
        pytest.skip("no candidate left to pick")
    E = workloads.gaussian_table(N, D, seed=seed) if seed % 2 else \
        workloads.clustered_table(N, D, n_centres=8, seed=seed)
    if mask is not None:
        # every sequence must have L candidates left
        avail = N - int(mask.sum()) - (mask[starts] == 0).astype(int)
        L = int(min(L, avail.min()))
        if L < 1:
            pytest.skip("no candidate left to pick")
    tr = np.unique(np.linspace(0, B - 1, num=min(B, 4)).astype(np.int32))
    picks, trace = _run(es, E, starts, L, mask, tr, pair=pair)
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, tr)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("variant", ["fp16", "centroid", "fp16-centroid"])
def test_random_shapes_variants(es, seed, variant):
    """The random shapes above on fp16 storage (tables of fp16 numbers) and
    on the centroid criterion, against the oracle."""
    N, D, B, L, mask, starts = _random_case(seed)
    if L == 0:
        pytest.skip("no candidate left to pick")
    E = workloads.clustered_table(N, D, n_centres=8, seed=seed)
    if variant.startswith("fp16"):
        E = _fp16_table(E)
    if mask is not None:
        avail = N - int(mask.sum()) - (mask[starts] == 0).astype(int)
        L = int(min(L, avail.min()))
        if L < 1:
            pytest.skip("no candidate left to pick")
    tr = np.unique(np.linspace(0, B - 1, num=min(B, 4)).astype(np.int32))
    if variant == "fp16":
        picks, trace = _run(es, E, starts, L, mask, tr, storage=1)
        check_picks_valid(starts, mask, picks, N)
        check_dseq_teacher_forced(E, starts, mask, picks, trace, tr)
    else:
        picks, trace = _run(es, E, starts, L, mask, tr, criterion=1,
                            storage=1 if variant == "fp16-centroid" else 0)
        check_picks_valid(starts, mask, picks, N)
        check_centroid_teacher_forced(E, starts, mask, picks, trace, tr)


def test_resume_without_state_rejected(es):
    E = workloads.gaussian_table(64, 16, seed=3)
    ctx = es.dseq_create(torch.from_numpy(E).cuda())
    try:
        es.dseq_set_option("resume", 1, ctx)
        with pytest.raises(es.DseqError):
            es.dseq_run(ctx, torch.tensor([0, 5], dtype=torch.int32, device="cuda"), 3)
    finally:
        ctx.close()


# --------------------------------------------------------------------------
# The Gram engine (max-min on split storage): the table's Gram matrix on the
# tensor cores, then one row of it per sequence and iteration, against the
# same oracle under the same teacher-forced tolerances.


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_gram_small_teacher_forced(es, case):
    N, D, B, L, kind, frac = case
    E = workloads.gaussian_table(N, D, seed=N) if kind == "gaussian" else \
        workloads.clustered_table(N, D, n_centres=16, seed=N)
    starts = workloads.starts(N, B, seed=N)
    mask = None
    if frac > 0:
        rng = np.random.default_rng(N)
        mask = (rng.random(N) < frac).astype(np.uint8)
        mask[starts[: B // 3]] = 1  # some starts are masked themselves
    trace_seqs = np.arange(B, dtype=np.int32) if B <= 200 else \
        np.sort(np.random.default_rng(1).choice(B, 64, replace=False)).astype(np.int32)
    picks, trace = _run(es, E, starts, L, mask, trace_seqs, gram=1)
    assert es.dseq_last_stat("gram") == 1
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, trace_seqs)


@pytest.mark.parametrize("case", EXTREME, ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_gram_extreme_shapes_teacher_forced(es, case):
    N, D, B, L = case
    E = workloads.gaussian_table(N, D, seed=D + N)
    starts = workloads.starts(N, B, seed=D + N)
    tr = np.unique(np.array([0, B // 2, B - 1], np.int32))
    picks, trace = _run(es, E, starts, L, None, tr, gram=1)
    check_picks_valid(starts, None, picks, N)
    check_dseq_teacher_forced(E, starts, None, picks, trace, tr)


def _walk_run(es, E, starts, L, mask, tr, walk):
    es.dseq_set_option("walk", walk)
    picks, trace = _run(es, E, starts, L, mask, tr, gram=1)
    assert es.dseq_last_stat("gram") == 1
    return picks, trace, es.dseq_last_stat("walk")


def test_gram_running_minima_too_long_for_one_cta(es):
    """A table whose running-minimum rows (120 KB) are too long for one CTA's
    shared memory (masked rows, ragged N): by default the walk spreads them
    over a cluster of CTAs; in global memory (walk = 3) it gives the same
    picks and minima, bit for bit; one CTA (walk = 1) is refused."""
    N, D, B, L = 30011, 48, 37, 10
    E = workloads.clustered_table(N, D, n_centres=20, seed=31)
    starts = workloads.starts(N, B, seed=31)
    mask = (np.random.default_rng(31).random(N) < 0.05).astype(np.uint8)
    tr = np.arange(B, dtype=np.int32)
    picks, trace, place = _walk_run(es, E, starts, L, mask, tr, 0)
    assert place == 2
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, tr)
    picks_g, trace_g, place = _walk_run(es, E, starts, L, mask, tr, 3)
    assert place == 3
    assert np.array_equal(picks_g, picks)
    assert np.array_equal(trace_g, trace)
    with pytest.raises(es.DseqError):
        _walk_run(es, E, starts, L, mask, tr, 1)


@pytest.mark.parametrize("case", [(1000, 96, 200, 16), (3001, 40, 29, 12), (37, 5, 9, 20),
                                  (2048, 8, 5, 6), (2049, 8, 5, 6), (4608, 8, 5, 6),
                                  (4609, 24, 7, 9), (8704, 24, 7, 9), (8705, 24, 7, 9),
                                  (12288, 16, 6, 9), (24576, 16, 6, 9), (24600, 16, 6, 9),
                                  (32768, 8, 4, 5), (40000, 16, 6, 7), (65537, 8, 3, 4),
                                  (140000, 16, 4, 5)],
                         ids=lambda c: f"N{c[0]}_D{c[1]}_B{c[2]}_L{c[3]}")
def test_gram_walk_places_identical(es, case):
    """The three places of the running minima (one CTA: in its registers up
    to N = 8704, else in its shared memory; a cluster's shared memory;
    global memory) run the same arithmetic in the same order per candidate:
    identical picks and traced minima, and the oracle's.  Rows shorter than
    the cluster (N = 37: some CTAs hold no candidate), every one-CTA shape
    and its boundaries (registers: 4, 9 and 17 vectors per thread, N = 2048
    / 2049 and 4608 / 4609 where the shape changes, N = 8704 the last row of
    the widest; shared memory from N = 8705, a row
    of exactly 48 KB at N = 12288, whose launch needs the raised shared
    memory limit once the static reduction slots are added, the largest
    one-CTA row N = 24576), and every cluster shape: up to 1,024
    vectors per CTA (exactly 1,024 at N = 32768), up to 2,048 (N = 40000),
    beyond (N = 65537), and more than one batch of loads per CTA
    (N = 140000, 78 GB of G) included."""
    N, D, B, L = case
    E = workloads.gaussian_table(N, D, seed=N + 7)
    starts = workloads.starts(N, B, seed=N + 7)
    mask = (np.random.default_rng(N).random(N) < 0.03).astype(np.uint8)
    mask[starts[:2]] = 1
    tr = np.unique(np.array([0, B // 2, B - 1], np.int32))
    out = {}
    for walk in (1, 2, 3):
        if walk == 1 and 4 * ((N + 31) // 32 * 32) > 96 * 1024:
            continue
        out[walk] = _walk_run(es, E, starts, L, mask, tr, walk)
        assert out[walk][2] == walk
    ref = out[min(out)]
    check_picks_valid(starts, mask, ref[0], N)
    check_dseq_teacher_forced(E, starts, mask, ref[0], ref[1], tr)
    for walk, (picks, trace, _) in out.items():
        assert np.array_equal(picks, ref[0]), f"walk={walk}"
        assert np.array_equal(trace, ref[1]), f"walk={walk}"
    # the walk kernels without the trace branch (a separate instantiation)
    for walk in out:
        es.dseq_set_option("walk", walk)
        picks, _ = _run(es, E, starts, L, mask, None, gram=1)
        assert es.dseq_last_stat("gram") == 1 and es.dseq_last_stat("walk") == walk
        assert np.array_equal(picks, ref[0]), f"untraced walk={walk}"
    es.dseq_set_option("walk", 0)


@pytest.mark.parametrize("N,place", [(8704, 1), (16384, 1), (16385, 2)])
def test_gram_default_place(es, N, place):
    """The default place of the running minima follows the row length: one
    CTA up to 64 KB of minima (N = 16384; in registers up to N = 8704),
    the cluster beyond; same picks as the global-memory walk."""
    D, B, L = 16, 5, 6
    E = workloads.gaussian_table(N, D, seed=N)
    starts = workloads.starts(N, B, seed=N)
    es.dseq_set_option("walk", 0)
    picks, _ = _run(es, E, starts, L, None, None, gram=1)
    assert es.dseq_last_stat("gram") == 1 and es.dseq_last_stat("walk") == place
    es.dseq_set_option("walk", 3)
    picks_g, _ = _run(es, E, starts, L, None, None, gram=1)
    assert es.dseq_last_stat("walk") == 3
    es.dseq_set_option("walk", 0)
    assert np.array_equal(picks, picks_g)


def test_gram_worked_examples(es):
    """The square of four unit vectors and the orthonormal table (every
    off-diagonal distance 1: a pure tie-break) on the Gram engine."""
    E = np.array([[1, 0], [0, 1], [-1, 0], [0, -1]], np.float32)
    picks, _ = _run(es, E, np.array([0], np.int32), 3, gram=1)
    assert picks.tolist() == [[2, 1, 3]]
    N = 40
    E = np.eye(N, dtype=np.float32)
    starts = np.array([0, 7, 39], np.int32)
    picks, _ = _run(es, E, starts, N - 1, gram=1)
    for b, s0 in enumerate(starts):
        assert picks[b].tolist() == [c for c in range(N) if c != s0]


@pytest.mark.parametrize("seed", range(8))
def test_gram_random_shapes_teacher_forced(es, seed):
    N, D, B, L, mask, starts = _random_case(seed)
    if L == 0:
        pytest.skip("no candidate left to pick")
    E = workloads.gaussian_table(N, D, seed=seed) if seed % 2 else \
        workloads.clustered_table(N, D, n_centres=8, seed=seed)
    if mask is not None:
        avail = N - int(mask.sum()) - (mask[starts] == 0).astype(int)
        L = int(min(L, avail.min()))
        if L < 1:
            pytest.skip("no candidate left to pick")
    tr = np.unique(np.linspace(0, B - 1, num=min(B, 4)).astype(np.int32))
    picks, trace = _run(es, E, starts, L, mask, tr, gram=1)
    check_picks_valid(starts, mask, picks, N)
    check_dseq_teacher_forced(E, starts, mask, picks, trace, tr)


def test_gram_automatic_choice(es):
    """gram = 2 (the default): the Gram engine where sequences make many more
    picks than the table has rows, the per-iteration kernel where they do not."""
    cfg = workloads.DIVERSITY["tiny"]
    _run(es, cfg.table(seed=0), cfg.starts(seed=0), cfg.L, gram=2)
    assert es.dseq_last_stat("gram") == 0
    N, D, B, L = 2000, 768, 1500, 40
    E = workloads.clustered_table(N, D, n_centres=10, seed=3)
    picks, _ = _run(es, E, workloads.starts(N, B, seed=3), L, gram=2)
    assert es.dseq_last_stat("gram") == 1
    assert es.dseq_last_stat("gram_ns") > 0 and es.dseq_last_stat("walk_ns") > 0


@pytest.mark.parametrize("name", ["page1", "n32k", "scale"])
def test_gram_full_size_teacher_forced(es, name):
    """The full configurations on the engine the library picks for them (the
    Gram engine), the benchmark's launch configuration, with a seeded subset
    of sequences followed by the oracle."""
    cfg = workloads.DIVERSITY[name]
    E = cfg.table(seed=0)
    starts = cfg.starts(seed=0)
    tr = np.sort(np.random.default_rng(0).choice(cfg.B, cfg.oracle_seqs, replace=False))
    picks, trace = _run(es, E, starts, cfg.L, trace_seqs=tr.astype(np.int32), gram=2)
    assert es.dseq_last_stat("gram") == 1
    check_dseq_teacher_forced(E, starts[tr], None, picks[tr], trace, np.arange(tr.size))
    assert np.all((picks >= 0) & (picks < cfg.N))
    srt = np.sort(picks, axis=1)
    assert not np.any(srt[:, 1:] == srt[:, :-1]), "a sequence repeats a pick"
    assert not np.any(picks == starts[:, None]), "a sequence picks its start"


@pytest.mark.parametrize("gram", [0, 1])
def test_buffer_cache(es, gram):
    """Destroyed contexts' buffers are kept for reuse (up to cache_mb per
    device): repeated create / run / destroy cycles from host arrays give
    identical picks and, once the cache holds their buffers, map no new
    device memory; with cache_mb = 0 every buffer is freed.  On the scan and
    on the Gram engine."""
    es.dseq_set_option("gram", gram)
    N, D, B, L = 3000, 64, 40, 12
    E = workloads.gaussian_table(N, D, seed=5)
    starts = workloads.starts(N, B, seed=5)

    def cycle():
        ctx = es.dseq_create(E)  # host arrays: every device buffer is the library's
        try:
            return np.array(es.dseq_run(ctx, starts, L))
        finally:
            ctx.close()

    def free_bytes():
        torch.cuda.synchronize()
        return torch.cuda.mem_get_info()[0]

    try:
        cycle()  # modules loaded, one-time set-up done
        es.dseq_set_option("cache_mb", 0)
        assert es.dseq_get_option("cache_mb") == 0
        free0 = free_bytes()
        p0 = cycle()
        assert free_bytes() == free0, "cache_mb = 0 kept device memory"
        es.dseq_set_option("cache_mb", -1)
        p1 = cycle()
        free1 = free_bytes()
        assert free1 < free0, "no buffer was kept"
        p2 = cycle()
        assert free_bytes() == free1, "a cycle mapped new memory despite the cache"
        assert np.array_equal(p0, p1) and np.array_equal(p0, p2)
        es.dseq_set_option("cache_mb", 0)  # trims the cache
        assert free_bytes() == free0
    finally:
        es.dseq_set_option("cache_mb", -1)


def test_centroid_stays_on_the_scan(es):
    """The centroid criterion always runs the scan (its exact centroid
    sums), even with gram = 1."""
    E = workloads.gaussian_table(600, 32, seed=4)
    _run(es, E, np.array([0, 9], np.int32), 5, criterion=1, gram=1)
    assert es.dseq_last_stat("gram") == 0


def test_gram_full_ordering_page1_in_chunks(es):
    """The page-1 table ordered completely (L = N - 1) by every sequence on
    the Gram engine: each sequence is a permutation of the table, and four
    resumed chunks give the picks of one call; a seeded subset of sequences
    follows the oracle over the first iterations."""
    cfg = workloads.DIVERSITY["page1"]
    E = cfg.table(seed=0)
    starts = cfg.starts(seed=0)[:512]
    L = cfg.N - 1
    es.dseq_set_option("gram", 1)
    ctx = es.dseq_create(torch.from_numpy(E).cuda())
    try:
        st = torch.from_numpy(starts).cuda()
        whole = es.dseq_run(ctx, st, L).cpu().numpy()
        assert es.dseq_last_stat("gram") == 1
        parts = []
        for i, chunk in enumerate((2000, 1, 3000, L - 5001)):
            es.dseq_set_option("resume", 0 if i == 0 else 1, ctx)
            parts.append(es.dseq_run(ctx, st, chunk).cpu().numpy())
    finally:
        ctx.close()
    assert np.array_equal(np.concatenate(parts, axis=1), whole)
    full = np.sort(np.concatenate([starts[:, None], whole], axis=1), axis=1)
    assert np.array_equal(full, np.broadcast_to(np.arange(cfg.N), full.shape))
    tr = np.array([0, 255, 511], np.int32)
    picks, trace = _run(es, E, starts, 24, trace_seqs=tr, gram=1)
    assert np.array_equal(picks, whole[:, :24])
    check_dseq_teacher_forced(E, starts[tr], None, picks[tr], trace, np.arange(tr.size))

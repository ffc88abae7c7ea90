"""World-size-2 gloo tests of the host-side sharding: each rank takes its
contiguous share of sequences (or samples), computes it, and the gathered
result must equal the single-process result.  The per-rank compute here is
the CPU oracle (no GPU on this path); on GPUs each rank runs the library on
its own device with the same sharding."""
from __future__ import annotations

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from embedding_similarity_scan_gb300.shard import gather_rows, shard_range  # noqa: E402


def test_shard_range_covers_exactly():
    for total in (0, 1, 7, 3584, 8192):
        for world in (1, 2, 3, 8):
            spans = [shard_range(total, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == total
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [hi - lo for lo, hi in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_range(10, 2, 2)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import oracle
    import workloads

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        E = workloads.clustered_table(400, 24, n_centres=8, seed=3)
        starts = workloads.starts(400, 37, seed=3)
        lo, hi = shard_range(starts.size, rank, world)
        picks, _, _ = oracle.dseq(E, starts[lo:hi], 12, threads=1)
        all_picks = gather_rows(picks)
        X = workloads.bmu_samples(101, 16, seed=4)
        W = workloads.codebook(300, 16, seed=4)
        lo, hi = shard_range(X.shape[0], rank, world)
        idx, _, _ = oracle.bmu(X[lo:hi], W, threads=1)
        all_idx = gather_rows(idx)
        if rank == 0:
            np.save(os.path.join(out_dir, "picks.npy"), all_picks)
            np.save(os.path.join(out_dir, "idx.npy"), all_idx)
    finally:
        dist.destroy_process_group()


def test_two_rank_gather_equals_single_process(tmp_path):
    import oracle
    import workloads

    oracle.build()
    mp.spawn(_worker, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    E = workloads.clustered_table(400, 24, n_centres=8, seed=3)
    starts = workloads.starts(400, 37, seed=3)
    want, _, _ = oracle.dseq(E, starts, 12, threads=1)
    assert np.array_equal(np.load(tmp_path / "picks.npy"), want)
    X = workloads.bmu_samples(101, 16, seed=4)
    W = workloads.codebook(300, 16, seed=4)
    want_idx, _, _ = oracle.bmu(X, W, threads=1)
    assert np.array_equal(np.load(tmp_path / "idx.npy"), want_idx)

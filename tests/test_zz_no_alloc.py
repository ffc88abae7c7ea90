"""bmu_search_noalloc: the BMU search for callers that cannot allocate device
memory (a framework whose pooling allocator already holds nearly all of the
GPU's memory, or a latency-critical loop that cannot absorb the device-wide
synchronisation cudaMalloc may imply).  It runs on a fixed scratch array
inside the library instead of a growing workspace.

Called through the C ABI twice in a row on different inputs, each result
must match the allocating entry point, bmu_search, within the tolerances of
the BMU parity tests.  This file sorts last so that a run stopping at the
first failure has run every other test before it.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TOL = 1e-5


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from embedding_similarity_scan_gb300 import build as esb

    esb.build()
    import embedding_similarity_scan_gb300 as es

    return es.load()


def _call_noalloc(lib, X, W):
    n, D = X.shape
    idx = torch.full((n,), -7, dtype=torch.int32, device="cuda")
    dist = torch.full((n,), -7.0, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.bmu_search_noalloc(X.data_ptr(), n, W.data_ptr(), W.shape[0], D, idx.data_ptr(),
                                dist.data_ptr(), ctypes.c_void_p(stream))
    assert rc == 0, lib.dseq_last_error().decode()
    return idx, dist


def _call_reference(lib, X, W):
    n, D = X.shape
    idx = torch.empty((n,), dtype=torch.int32, device="cuda")
    dist = torch.empty((n,), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.bmu_search(X.data_ptr(), n, W.data_ptr(), W.shape[0], D, idx.data_ptr(),
                        dist.data_ptr(), ctypes.c_void_p(stream))
    assert rc == 0, lib.dseq_last_error().decode()
    return idx, dist


def _agree(X, W, got, ref):
    """Same neuron, or a neuron at the same distance within the tolerance;
    distances within 1e-5 * (|x|^2 + |w|^2)."""
    X64 = X.cpu().numpy().astype(np.float64)
    W64 = W.cpu().numpy().astype(np.float64)
    gi, gd = got[0].cpu().numpy(), got[1].cpu().numpy().astype(np.float64)
    ri, rd = ref[0].cpu().numpy(), ref[1].cpu().numpy().astype(np.float64)
    assert np.all((gi >= 0) & (gi < W64.shape[0]))
    scale = (X64 ** 2).sum(1) + (W64[ri] ** 2).sum(1)
    same = gi == ri
    close = np.abs(gd - rd) <= TOL * scale
    assert np.all(same | close), f"{np.count_nonzero(~(same | close))} indices differ"
    assert np.all(close), f"distances differ by up to {np.abs(gd - rd).max()}"


def test_noalloc_matches_bmu_search_on_two_calls_in_a_row(lib):
    # D <= 256 runs the resident-sample kernel, D = 300 the streaming one
    cases = [(3000, 5000, 96, 1), (1700, 9000, 200, 2), (1000, 2000, 300, 3)]
    inputs = []
    for n, M, D, seed in cases:
        X = torch.from_numpy(workloads.bmu_samples(n, D, seed=seed)).cuda()
        W = torch.from_numpy(workloads.codebook(M, D, seed=seed)).cuda()
        inputs.append((X, W))
    # two calls in a row on the shared scratch, then the allocating entry point
    results = [_call_noalloc(lib, X, W) for X, W in inputs]
    torch.cuda.synchronize()
    for (X, W), got in zip(inputs, results):
        ref = _call_reference(lib, X, W)
        _agree(X, W, got, ref)
        # the same kernels on the same split operands: the same bits
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])


def test_warmed_call_allocates_nothing(lib):
    """After a first call (the one-time set-up), a call leaves the device's
    free memory and torch's allocator exactly as they were."""
    X = torch.from_numpy(workloads.bmu_samples(2000, 128, seed=4)).cuda()
    W = torch.from_numpy(workloads.codebook(3000, 128, seed=4)).cuda()
    first = _call_noalloc(lib, X, W)
    idx = torch.empty((X.shape[0],), dtype=torch.int32, device="cuda")
    dist = torch.empty((X.shape[0],), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.bmu_search_noalloc(X.data_ptr(), X.shape[0], W.data_ptr(), W.shape[0], X.shape[1],
                                idx.data_ptr(), dist.data_ptr(), ctypes.c_void_p(stream))
    assert rc == 0, lib.dseq_last_error().decode()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.equal(idx, first[0]) and torch.equal(dist, first[1])


def test_noalloc_rejects_memory_of_another_device(lib):
    """Inputs on a GPU other than the current one are rejected before any
    work is enqueued (needs two GPUs)."""
    if torch.cuda.device_count() < 2:
        pytest.skip("one GPU: no memory of another device to pass")
    X = torch.zeros((4, 8), dtype=torch.float32, device="cuda:1")
    W = torch.ones((6, 8), dtype=torch.float32, device="cuda:0")
    idx = torch.empty(4, dtype=torch.int32, device="cuda:0")
    dist = torch.empty(4, dtype=torch.float32, device="cuda:0")
    with torch.cuda.device(0):
        rc = lib.bmu_search_noalloc(X.data_ptr(), 4, W.data_ptr(), 6, 8, idx.data_ptr(),
                                    dist.data_ptr(), None)
    assert rc == -1 and "device 1" in lib.dseq_last_error().decode()


def test_noalloc_rejects_what_it_cannot_serve(lib):
    X = torch.zeros((4, 8), dtype=torch.float32, device="cuda")
    W = torch.ones((6, 8), dtype=torch.float32, device="cuda")
    idx = torch.empty(4, dtype=torch.int32, device="cuda")
    dist = torch.empty(4, dtype=torch.float32, device="cuda")
    # host outputs: nothing may be staged
    host_idx = np.empty(4, np.int32)
    rc = lib.bmu_search_noalloc(X.data_ptr(), 4, W.data_ptr(), 6, 8, host_idx.ctypes.data,
                                dist.data_ptr(), None)
    assert rc == -1 and "device memory" in lib.dseq_last_error().decode()
    # more scratch than the fixed array holds: rejected before any GPU work
    big_n = 200_000
    Xb = torch.empty((1, 256), dtype=torch.float32, device="cuda")
    rc = lib.bmu_search_noalloc(Xb.data_ptr(), big_n, W.data_ptr(), 6, 256, idx.data_ptr(),
                                dist.data_ptr(), None)
    assert rc == -1 and "scratch" in lib.dseq_last_error().decode()
    # a valid call still works afterwards
    got = _call_noalloc(lib, X, W)
    _agree(X, W, got, _call_reference(lib, X, W))

"""Host-side helpers of bench.py (no GPU): the launch-variant key of the
traffic lookup, the walk kernel named for a run's place and table size,
and that a profile summary's traffic is taken only from the section whose
source hash is the current kernel source's."""
from __future__ import annotations

import bench


def test_traffic_variant_keys():
    assert bench._traffic_variant([]) == ""
    assert bench._traffic_variant(["pair=0"]) == "_pair0"
    assert bench._traffic_variant(["pair=0", "criterion=1"]) == "_pair0_centroid"
    assert bench._traffic_variant(["storage=1", "pair=0"]) == "_pair0_f16"
    assert bench._traffic_variant(["criterion=1", "storage=1", "pair=0"]) == "_pair0_centroid_f16"
    assert bench._traffic_variant(["storage=1"]) == "_f16"


def test_walk_kernel_names():
    # one CTA: registers up to 8704 candidates, shared memory beyond
    assert bench._walk_kernel_name(1, 8359) == "gram_walk_kernel_regs"
    assert bench._walk_kernel_name(1, 8704) == "gram_walk_kernel_regs"
    assert bench._walk_kernel_name(1, 8705) == "gram_walk_kernel"
    assert bench._walk_kernel_name(2, 131072) == "gram_walk_cluster_kernel"
    assert bench._walk_kernel_name(3, 300000) == "gram_walk_kernel"
    # every name has its sources listed for the profile lookup
    for name in ("gram_walk_kernel_regs", "gram_walk_kernel", "gram_walk_cluster_kernel"):
        assert name in bench.KERNEL_SOURCES


def test_profiled_traffic_uses_the_current_source_section(tmp_path, monkeypatch):
    current = bench._kernel_hash("tc_dseq_kernel")
    stale = "0" * 16 if current != "0" * 16 else "1" * 16
    (tmp_path / "tc_dseq_kernel.demo.md").write_text(
        f"kernel_source_sha256_16: {stale}\n\ntraffic_bytes_per_launch_pair0: 1.0e9\n\n"
        f"kernel_source_sha256_16: {current}\n\ntraffic_bytes_per_launch_pair0: 2.5e9\n"
        f"traffic_bytes_per_launch_pair0_centroid: 3.0e8\n")
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench._profiled_traffic("tc_dseq_kernel", "demo", "_pair0") == 2.5e9
    assert bench._profiled_traffic("tc_dseq_kernel", "demo", "_pair0_centroid") == 3.0e8
    # a variant the current section does not list, and a workload without a file
    assert bench._profiled_traffic("tc_dseq_kernel", "demo", "_pair0_f16") is None
    assert bench._profiled_traffic("tc_dseq_kernel", "other", "_pair0") is None


def test_profiled_traffic_ignores_stale_sections(tmp_path, monkeypatch):
    (tmp_path / "tc_dseq_kernel.demo.md").write_text(
        "kernel_source_sha256_16: ffffffffffffffff\n\ntraffic_bytes_per_launch_pair0: 1.0e9\n")
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    if bench._kernel_hash("tc_dseq_kernel") != "ffffffffffffffff":
        assert bench._profiled_traffic("tc_dseq_kernel", "demo", "_pair0") is None

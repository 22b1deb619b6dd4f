"""Host-side logic of bench.py (no GPU): the per-kernel source hashes that decide whether a committed
ncu traffic capture still applies, and the timing helpers' arithmetic."""
import importlib.util
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_every_kernel_kind_hashes_existing_sources(bench):
    csrc = os.path.join(ROOT, "communication_overlap_domino_gb300", "csrc")
    for kind, files in bench.KERNEL_SOURCES.items():
        assert all(os.path.exists(os.path.join(csrc, f)) for f in files), kind
        assert len(bench.kernel_source_hash(kind)) == 16
    # kernels built from the same files share a hash; different kernels do not
    assert bench.kernel_source_hash("gemm1") == bench.kernel_source_hash("bwd_dw")
    assert len({bench.kernel_source_hash(k) for k in ("fused", "gemm1", "shard_sum", "attn")}) == 4


def test_traffic_record_entries_are_well_formed(bench):
    with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
        rec = json.load(f)
    for key, entry in rec["kernels"].items():
        workload, kind = key.split("/")
        assert kind in bench.KERNEL_SOURCES, key
        assert entry["dram_bytes_per_launch"] > 0 and entry["algorithmic_bytes"] > 0
        assert "source_hash" in entry and entry["mu"] >= 1
        got = bench.ncu_traffic(kind, workload, entry["mu"])
        # a capture is reported exactly when its hash matches the kernel's current sources
        assert (got is not None) == (entry["source_hash"] == bench.kernel_source_hash(kind)), key
        # and only at the number of chunks it was captured at (a launch covers one chunk, or all of them)
        assert bench.ncu_traffic(kind, workload, 2 * entry["mu"]) is None, key


def test_traffic_lookup_rejects_unknown(bench):
    assert bench.ncu_traffic("no_such_kernel", "gpt_gelu_fwd", 2) is None
    assert bench.ncu_traffic("fused", "no_such_workload", 2) is None


def test_whole_job_throughput_counts_all_ranks(bench):
    # value = the units all ranks processed / the (max over ranks) time
    assert bench.whole_job_tflops(1e12, 4, 1000.0) == pytest.approx(4.0)

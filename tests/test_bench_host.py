"""Host-side helpers of bench.py (no GPU): the workload selection and the
reading of DRAM traffic from a committed ncu summary, which must be dropped
once the kernel's sources no longer match the capture."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_workload_selection():
    w2 = bench._workload(4, 2)
    assert (w2.T, w2.H, w2.Hkv, w2.d) == (4 * 4096, 16, 16, 128) and w2.seqlens == [4096] * 4
    small = bench._workload(3, 2)
    assert small.seqlens == [4096] * 3 and small.H == 16
    w5 = bench._workload(4, 5)
    assert (w5.T, w5.H, w5.Hkv) == (2 * 65536, 32, 8)
    w3 = bench._workload(4, 3)
    assert w3.T == 8 * 16384 and sum(w3.seqlens) == w3.T and w3.outlier_channels == 2
    # the mixed-path workload and its one-row case for profiler captures: the
    # same documents as the full workload's first 32768-token row
    w4 = bench._workload(4, 4)
    one = bench._workload(1, 4)
    assert w4.T == 4 * 32768 and one.T == 32768 and sum(one.seqlens) == one.T
    n = 0
    for i, length in enumerate(w4.seqlens):
        n += length
        if n == 32768:
            assert one.seqlens == w4.seqlens[:i + 1]
            break
    else:
        raise AssertionError("no row boundary at 32768 tokens")
    assert (one.H, one.Hkv, one.d, one.outlier_channels, one.seed) == (16, 16, 128, 2, w4.seed)


def _fake_profile(tmp_path, kernel, source_hash, full_bytes):
    d = tmp_path / "profiles"
    d.mkdir(exist_ok=True)
    (d / f"{kernel}_batched_4x4096.md").write_text(
        f"# {kernel}\n\nsource_hash: {source_hash}\n\n"
        f"dram_bytes_per_launch_capture: 1\ndram_bytes_per_launch_full_workload: {full_bytes}\n")


def test_profiled_traffic_matches_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "abc123")
    _fake_profile(tmp_path, "bwd_kernel", "abc123", 1234567)
    assert bench._profiled_traffic("bwd_kernel") == pytest.approx(1234567.0)


def test_profiled_traffic_dropped_when_sources_changed(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "def456")
    _fake_profile(tmp_path, "bwd_kernel", "abc123", 1234567)
    assert bench._profiled_traffic("bwd_kernel") is None


def test_profiled_traffic_missing_summary(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._profiled_traffic("fwd_kernel") is None


def test_kernel_source_hash_covers_the_kernel_sources():
    # every listed source exists, and the hash is stable across calls
    for k, files in bench.KERNEL_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(ROOT, "precision_causal_attention_token_gb300", "csrc", f)), f
        assert bench.kernel_source_hash(k) == bench.kernel_source_hash(k)

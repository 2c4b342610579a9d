"""Host-side pieces of bench.py (CPU only): the algorithmic FLOP and byte
counts of the layer block against the figures the workload table states,
and the rule that the recorded DRAM traffic is reported only while the GEMM
sources match the hash it was captured at."""
import os

import pytest

import bench


def test_block_flops_and_weight_bytes():
    # 2 T (QKV 7168x5120 + O 5120x5120 + gate/up 2x17408x5120 + down 5120x17408)
    assert bench.block_flops(1024) == 2 * 1024 * 330_301_440
    assert round(bench.block_flops(1024) / 1e9, 1) == 676.5
    # codes (1/2 byte) + scales (1/16 byte) per weight element: 185.8 MB
    assert bench.weight_bytes() == 330_301_440 // 2 + 330_301_440 // 16
    assert round(bench.weight_bytes() / 1e6, 1) == 185.8


def write_profile(root, sha, traffic="108074752"):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "gemm_swiglu_T1024.txt"), "w") as f:
        f.write("# command: ncu ... (comment lines may hold colons)\n")
        f.write(f"source_sha256: {sha}\n")
        f.write(f"traffic_bytes_per_launch: {traffic}\n")


def test_recorded_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0123456789abcdef")
    assert bench.recorded_traffic() is None                      # no summary
    write_profile(str(tmp_path), "0123456789abcdef")
    assert bench.recorded_traffic() == 108074752
    write_profile(str(tmp_path), "fedcba9876543210")
    assert bench.recorded_traffic() is None                      # the kernel changed since
    write_profile(str(tmp_path), "0123456789abcdef", traffic="n/a")
    assert bench.recorded_traffic() is None


def test_kernel_source_hash_covers_the_gemm_sources():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    assert h == bench.kernel_source_hash()

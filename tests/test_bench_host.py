"""Host logic of bench.py that the roofline fields depend on (no GPU)."""

import os

import bench


def write(path, text):
    with open(path, "w", encoding="utf-8") as f:
        f.write(text)


def test_kernel_source_hash_follows_the_include_closure(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    write(tmp_path / "k.cu", '#include "a.cuh"\n#include <cstdint>\n__global__ void k() {}\n')
    write(tmp_path / "a.cuh", '#pragma once\n#include "b.cuh"\n')
    write(tmp_path / "b.cuh", "#pragma once\nint b;\n")
    write(tmp_path / "other.cuh", "int other;\n")
    h0 = bench.kernel_source_hash("k.cu")
    write(tmp_path / "other.cuh", "int other2;\n")  # not included: same hash
    assert bench.kernel_source_hash("k.cu") == h0
    write(tmp_path / "b.cuh", "#pragma once\nint b2;\n")  # included transitively
    assert bench.kernel_source_hash("k.cu") != h0


def test_recorded_traffic_needs_a_matching_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "CSRC", str(tmp_path))
    write(tmp_path / "k.cu", "__global__ void k() {}\n")
    h = bench.kernel_source_hash("k.cu")
    rec = tmp_path / "rec.md"
    write(rec, f"# summary\n\n- source_hash: {h}\n- dram_bytes_per_launch: 12345\n")
    assert bench.recorded_traffic(str(rec), "k.cu") == 12345
    write(rec, "- source_hash: 0000000000000000\n- dram_bytes_per_launch: 12345\n")
    assert bench.recorded_traffic(str(rec), "k.cu") is None
    assert bench.recorded_traffic(str(tmp_path / "missing.md"), "k.cu") is None


def test_algorithmic_bytes_of_the_headline_workload():
    w = dict(B=256, gamma=7, V=128256, dtype="bf16")
    assert bench.logit_bytes(w) == 985_006_080      # (2 gamma + 1) rows per sequence
    assert bench.overlap_bytes(w) == 919_339_008    # 2 gamma rows per sequence
    assert bench.typical_bytes(w) == 525_336_576    # gamma + 1 rows per sequence
    assert bench.l2_note(bench.logit_bytes(w), "logits").startswith("inputs larger than L2")
    assert bench.l2_note(10_000_000, "x").startswith("inputs smaller than L2")


def test_committed_profiles_name_their_kernels():
    for path, unit in ((bench.TRAFFIC_FILE, bench.TRAFFIC_UNIT),
                       (bench.OVERLAP_TRAFFIC_FILE, "overlap.cu"),
                       (bench.TYPICAL_TRAFFIC_FILE, "chain_rows.cu")):
        assert os.path.exists(path)
        assert os.path.exists(os.path.join(bench.CSRC, unit))
        with open(path, encoding="utf-8") as f:
            text = f.read()
        assert "- source_hash:" in text and "- dram_bytes_per_launch:" in text
        assert "--clock-control none" in text


def test_all_core_oracle_baseline_matches_the_oracle_rows():
    # the all-core CPU baseline: spawned processes over shared memory, the
    # oracle's rows per second on a small chain workload
    from speculative_decoding_verification_temp_gb300 import workloads
    w = workloads.make_chain(3, 2, 300, dtype="f32", seed=5)
    rate, dt, procs, passes = bench.oracle_all_cores(w, 3)
    assert procs == min(3, os.cpu_count() or 1)
    assert rate > 0 and dt > 0 and passes == 1
    # the filtered workload of --op filters reaches the oracle's policy
    import numpy as np
    P = np.full(3, 0.5, np.float32)
    w["filters"] = dict(target_top_p=P, draft_top_p=P, target_min_p=P * 0.1, draft_min_p=P * 0.1)
    rate, dt, procs, passes = bench.oracle_all_cores(w, 3, min_s=0.05)
    assert rate > 0 and passes >= 1
    r1, _, _ = bench.oracle_sample_rate(w, 2)
    assert r1 > 0

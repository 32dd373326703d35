"""The benchmark's host-side arithmetic (CPU only): the algorithmic bytes it divides by, the
whole-job value, and the lookup of ncu traffic lines by the decode sources' hash."""
import sys
from pathlib import Path

import pytest

sys.path.insert(0, str(Path(__file__).resolve().parents[1]))
import bench  # noqa: E402
import kvsynth  # noqa: E402


def test_algorithmic_bytes_per_kernel_and_step():
    """Per launch: the scores read every cluster's mean key (bf16) and count, the estimation every
    value sum (fp32, or bf16) and count, the exact kernel the union rows x 512 B; per step also the
    queries (bf16) in and the outputs (fp32) out."""
    w = kvsynth.get_workload("llama3-8b-131k")
    U, C = w.units, w.clusters
    assert (U, C) == (8, 8192)
    rows, union = 75000.0, 0.93
    cand, step = bench.algorithmic_bytes(w, 4, rows, union)
    assert cand["scores"] == U * C * (128 * 2 + 4)
    assert cand["select_estimate"] == U * C * (128 * 4 + 4)
    assert cand["exact_merge"] == pytest.approx(rows * union * 512)
    assert step == pytest.approx(sum(cand.values()) + U * w.group * 128 * (2 + 4))
    cand16, _ = bench.algorithmic_bytes(w, 2, rows, union)
    assert cand16["select_estimate"] == U * C * (128 * 2 + 4)


def test_job_value_counts_every_rank_and_row():
    # 2 ranks x 100 steps x batch 16 x 1 layer in 0.5 s
    assert bench.job_value(2, 100, 16, 1, 0.5) == pytest.approx(6400.0)


def test_traffic_lines_follow_the_decode_sources(monkeypatch, tmp_path):
    """A traffic line counts only when its hash names the current decode sources."""
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "k_x.md").write_text(
        "traffic: kernel=k_exact_merge workload=wl source=0123456789abcdef dram_bytes_per_launch=4242\n"
        "traffic: kernel=k_exact_merge workload=other source=0123456789abcdef dram_bytes_per_launch=7\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "decode_source_hash", lambda: "0123456789abcdef")
    assert bench.ncu_traffic("k_exact_merge", "wl") == 4242
    assert bench.ncu_traffic("k_exact_merge", "other") == 7
    assert bench.ncu_traffic("k_scores", "wl") is None
    monkeypatch.setattr(bench, "decode_source_hash", lambda: "fedcba9876543210")
    assert bench.ncu_traffic("k_exact_merge", "wl") is None


def test_decode_source_hash_is_stable_and_sixteen_hex_digits():
    h = bench.decode_source_hash()
    assert h == bench.decode_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0

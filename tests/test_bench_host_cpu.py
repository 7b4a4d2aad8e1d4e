"""Host-side logic of the benchmark (CPU only): the nominal Newton-Schulz FLOP
count behind the TFLOP/s figures, the per-stage to per-family merge, and the
gate that reports a recorded DRAM traffic figure only while the kernel
sources it was measured on are unchanged."""
import os
import shutil

import pytest

import bench
from synth import workloads as W


def _nominal(m, n):
    """One quintic iteration on an m x n view, m <= n: 2m^2n (A = X X^T)
    + 2m^3 (A^2) + 2m^2n (the product with X), as the benchmark counts it."""
    return 4 * m * m * n + 2 * m ** 3


def test_ns_flops_of_the_7b_shape_step():
    # 32 layers of {Q, O 4096^2; K, V 1024 x 4096; gate_up as two 14336 x 4096
    # views; down 4096 x 14336}, five iterations each, written out by hand.
    per_layer = (2 * _nominal(4096, 4096) + 2 * _nominal(1024, 4096)
                 + 2 * _nominal(4096, 14336) + _nominal(4096, 14336))
    want = 32 * 5 * per_layer
    assert bench.ns_flops(W.llama7b()) == want
    assert want == pytest.approx(665.89e12, rel=1e-4)


def test_ns_flops_uses_the_short_side_and_counts_views():
    wl = W.Workload("t", muon=[W.MuonSpec("tall", 3, 96, 32, "f32", "f32"),
                               W.MuonSpec("wide", 1, 32, 96, "f32", "f32")],
                    adamw=[], muon_hp=dict(W.MUON_HP, ns_steps=2), adam_hp=dict(W.ADAM_HP))
    assert bench.ns_flops(wl) == 2 * (3 + 1) * _nominal(32, 96)


def test_family_stats_merges_stages():
    stats = {
        "ns_gemm.gram": dict(launches=2, total_ms=1.5, bytes=10.0, flops=4.0, flops_executed=2.0),
        "ns_gemm.apply": dict(launches=3, total_ms=0.5, bytes=5.0, flops=6.0, flops_executed=6.0),
        "adamw": dict(launches=1, total_ms=0.25, bytes=7.0, flops=0.0, flops_executed=0.0),
    }
    fam = bench.family_stats(stats)
    assert fam["ns_gemm"] == dict(launches=5, total_ms=2.0, bytes=15.0, flops=10.0,
                                  flops_executed=8.0)
    assert fam["adamw"]["launches"] == 1 and set(fam) == {"ns_gemm", "adamw"}


def _fake_root(tmp_path):
    csrc = tmp_path / "muon_adamw_hybrid_gb300" / "csrc"
    csrc.mkdir(parents=True)
    real = os.path.join(bench.ROOT, "muon_adamw_hybrid_gb300", "csrc")
    for files in bench.KERNEL_SOURCES.values():
        for f in files:
            shutil.copy(os.path.join(real, f), csrc / f)
    (tmp_path / "profiles").mkdir()
    return tmp_path


def test_traffic_record_is_dropped_once_its_sources_change(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    digest = bench.sources_digest("adamw")
    (root / "profiles" / "dram_toy.md").write_text(
        "text\n"
        f"traffic-record: kernel=adamw bytes_per_launch=1.5e+09 sources={digest}\n"
        "traffic-record: kernel=ns_gemm bytes_per_launch=2.0e+09 sources=0000000000000000\n"
        "traffic-record: kernel=unknown bytes_per_launch=3.0e+09 sources=0000000000000000\n")
    assert bench.traffic_records("toy") == {"adamw": 1.5e9}
    # any byte of any source of the family invalidates the record
    with open(root / "muon_adamw_hybrid_gb300" / "csrc" / "adamw.cu", "a") as f:
        f.write("\n")
    assert bench.sources_digest("adamw") != digest
    assert bench.traffic_records("toy") == {}


def test_missing_profile_gives_no_records(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(_fake_root(tmp_path)))
    assert bench.traffic_records("absent") == {}


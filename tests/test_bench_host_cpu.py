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
    assert bench.traffic_records("toy") == {"adamw": ("bytes", 1.5e9)}
    # any byte of any source of the family invalidates the record
    with open(root / "muon_adamw_hybrid_gb300" / "csrc" / "adamw.cu", "a") as f:
        f.write("\n")
    assert bench.sources_digest("adamw") != digest
    assert bench.traffic_records("toy") == {}


def test_missing_profile_gives_no_records(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(_fake_root(tmp_path)))
    assert bench.traffic_records("absent") == {}



def test_tensor_peak_follows_the_power_cap():
    peaks = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
    assert bench.tensor_peak(peaks, "measured", {"reasons": ["sw_power_cap"]})[0] == 1700.0
    assert bench.tensor_peak(peaks, "measured", {"reasons": []})[0] == 1900.0


def test_gemm_roofline_leads_with_executed_flops():
    peaks = {"bf16_tflops": 2000.0, "bf16_tflops_sustained": 1600.0, "hbm_gbs": 6800.0}
    v = dict(launches=4, total_ms=1000.0, bytes=8e9, flops=2.0e15, flops_executed=1.5e15)
    r = bench.gemm_roofline(v, peaks, "measured", {"reasons": ["sw_power_cap"]}, traffic=3e9)
    assert r["achieved"] == 1500.0 and r["frac"] == round(1500.0 / 1600.0, 4)
    assert r["nominal_tflops"] == 2000.0 and r["nominal_frac"] == 1.25
    assert r["frac_of_datasheet"] == round(1500.0 / bench.DATASHEET_BF16_TFLOPS, 4)
    assert r["algorithmic_bytes_per_launch"] == 2e9 and r["traffic"] == 3e9


def test_cpu_baseline_and_reference_arm_share_one_sample():
    for name in ("single", "gpt124m", "llama7b", "moe_mla", "adamw_2p30"):
        wl = W.WORKLOADS[name]()
        assert bench.oracle_plan(wl) == bench.oracle_plan(wl)
        views, adam = bench.oracle_plan(wl)
        assert sum(f for *_, f in views) <= bench.ORACLE_NS_FLOP_BUDGET
        assert sum(c for _, c in adam) <= bench.ORACLE_ADAM_ELEMS


def test_cpu_baseline_record_states_what_it_covers():
    wl = W.single_matrix()
    views, adam = bench.oracle_plan(wl)
    rec = bench.cpu_baseline_record(wl, views, adam, None, 0.01, 5.0)
    assert rec["extrapolated"] is False and rec["sample_fraction"]["ns_flops"] == 1.0
    wl = W.llama7b()
    views, adam = bench.oracle_plan(wl)
    rec = bench.cpu_baseline_record(wl, views, adam, None, 8.0, 1e6)
    assert rec["extrapolated"] is True
    assert 0 < rec["sample_fraction"]["ns_flops"] < 0.05
    assert rec["kind"] == "oracle" and rec["cores"] >= 1


def test_ratio_record_applies_to_named_workloads_and_scales(tmp_path, monkeypatch):
    root = _fake_root(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    digest = bench.sources_digest("ns_gemm")
    (root / "profiles" / "dram_slice.md").write_text(
        f"traffic-record: kernel=ns_gemm ratio=1.25 applies_to=big,slice sources={digest}\n")
    rec = bench.traffic_records("big")
    assert rec == {"ns_gemm": ("ratio", 1.25)}
    assert bench.traffic_for(rec, "ns_gemm", 8e9) == 1e10
    assert bench.traffic_for(rec, "adamw", 8e9) is None
    assert bench.traffic_records("other") == {}


def test_committed_traffic_records_are_well_formed():
    """Every traffic-record line under profiles/ names a kernel family the
    benchmark hashes, a ratio or a byte count in a plausible range, a
    16-hex-digit source digest, and only workloads the benchmark can run
    (a registered set or an NS-only point), so a typo cannot silently leave a
    configuration without its record."""
    import glob
    import os
    import re
    from synth import workloads as W
    paths = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "dram_*.md")))
    assert paths
    seen = 0
    for path in paths:
        for line in open(path):
            if not line.startswith("traffic-record:"):
                continue
            seen += 1
            kv = dict(tok.split("=", 1) for tok in line.split()[1:])
            assert kv["kernel"] in bench.KERNEL_SOURCES, (path, line)
            assert re.fullmatch(r"[0-9a-f]{16}", kv["sources"]), (path, line)
            if "ratio" in kv:
                assert 0.5 < float(kv["ratio"]) < 3.0, (path, line)
            else:
                assert float(kv["bytes_per_launch"]) > 0, (path, line)
            for w in kv["applies_to"].split(","):
                assert w in W.WORKLOADS or re.fullmatch(r"ns_(1:1|1:4|4:1)_n\d+_batch\d+", w), \
                    (path, w)
    assert seen >= 10

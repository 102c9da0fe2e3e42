"""Host-side helpers of bench.py on CPU: the clock record, the DRAM-traffic record that goes
stale with the kernel's sources, the roofline peak and its fallback, the JSON config, and the
reference arm's time budget."""
import json
import os
import shutil

import numpy as np
import pytest

import bench
from speculative_decoding_tree_mask_gb300 import workloads as W


def test_clock_summary_median_max_and_reasons():
    s = bench.ClockSampler(0)
    s.lines = [(float(i), ln) for i, ln in enumerate([
        "2070, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "1980, 2070, 1210.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2070, 2070, 1300.2, 0x0, Not Active, Not Active, Not Active, Not Active",
        "[N/A], 2070, 0, 0x0, Not Active, Not Active, Not Active, Not Active",   # unreadable
        "garbage",
    ])]
    out = s.summary()
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["samples"] == 3
    assert out["reasons"] == ["sw_power_cap"]
    s.lines.append((5.0, "1400, 2070, 1390, 0x8, Active, Not Active, Active, Not Active"))
    assert s.summary()["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]


def test_clock_summary_of_a_short_region_takes_the_bracketing_samples():
    """A timed region shorter than the sampling interval still gets the samples on both
    sides of it (within one interval); samples farther away are left out."""
    s = bench.ClockSampler(0, interval_ms=50)
    row = "{}, 2070, 1000, 0x0, Not Active, Not Active, Not Active, {}"
    s.lines = [(0.90, row.format(1000, "Active")), (0.98, row.format(2070, "Not Active")),
               (1.03, row.format(2060, "Not Active")), (1.20, row.format(1500, "Active"))]
    s.mark(1.00, 1.014)
    out = s.summary(region=True)
    assert out["samples"] == 2 and out["sm_mhz"] == 2065.0 and out["reasons"] == []
    assert s.summary()["samples"] == 4 and s.summary()["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples():
    out = bench.ClockSampler(0).summary()
    assert out == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                   "interval_ms": 50}


def _copy_tree(tmp_path):
    """A scratch copy of the kernel sources and the traffic record, with bench pointed at it."""
    root = tmp_path / "repo"
    shutil.copytree(os.path.join(bench.ROOT, "speculative_decoding_tree_mask_gb300", "csrc"),
                    root / "speculative_decoding_tree_mask_gb300" / "csrc")
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    return root


def test_traffic_record_goes_stale_with_its_sources(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    rec_path = root / "profiles" / "traffic.json"
    recs = json.loads(rec_path.read_text())
    rec = recs["row_stats.cu"]
    # a record taken from the current sources is reported
    rec["source_sha"] = bench.source_sha(rec["sources"])
    rec_path.write_text(json.dumps(recs))
    assert bench.traffic_record("row_stats.cu") == rec["bytes_per_launch"]
    # a comment edit leaves the kernel, and the record, as they were
    hdr = root / "speculative_decoding_tree_mask_gb300" / "csrc" / rec["sources"][-1]
    hdr.write_text(hdr.read_text() + "\n// a remark\n/* and\n another */\n")
    assert bench.traffic_record("row_stats.cu") == rec["bytes_per_launch"]
    # a code change in any of the kernel's files (a header included) makes it stale
    hdr.write_text(hdr.read_text() + "\nconstexpr int kEdited = 1;\n")
    assert bench.traffic_record("row_stats.cu") is None
    # kernels without a record, and no record file at all
    assert bench.traffic_record("no_such_kernel.cu") is None
    rec_path.unlink()
    assert bench.traffic_record("row_stats.cu") is None


def test_committed_traffic_record_names_existing_sources():
    recs = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for name, rec in recs.items():
        assert name in rec["sources"]
        for f in rec["sources"]:
            assert os.path.exists(os.path.join(bench.ROOT, "speculative_decoding_tree_mask_gb300",
                                               "csrc", f)), f
        assert rec["bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        assert rec["bytes_per_launch"] >= rec["algorithmic_bytes_per_launch"]


def test_peaks_measured_then_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    pk, kind = bench.peaks()
    assert kind == "fallback" and pk["hbm_gbs"] == bench.FALLBACK_HBM_GBS
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6779.7}))
    pk, kind = bench.peaks()
    assert kind == "measured" and pk["hbm_gbs"] == 6779.7


@pytest.mark.parametrize("world", [1, 4])
def test_config_names_the_workload(world):
    w = W.WORKLOADS[bench.WORKLOAD]
    cfg = bench.config_of(w, world)
    assert cfg["workload"].startswith("large_tree: B=256 N=64 V=152064 bf16")
    assert cfg["global_batch"] == 256 * world
    assert cfg["nodes_per_request"] == 64 and cfg["vocab"] == 152064
    assert "4.98 GB" in cfg["l2"]
    assert not {"model", "seq_len"} & set(cfg)
    assert bench.aggregate_throughput(world, w.draft_nodes, 0.5) == world * 256 * 63 / 5e-4


def test_reference_arm_samples_requests_to_its_budget(monkeypatch, capsys):
    """The reference arm (the oracle) keeps its whole run near its time budget: past it, each
    step verifies only the first requests of the batch, and the line says how many."""
    import argparse
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    args = argparse.Namespace(requests=3, steps=2, warmup=1)
    monkeypatch.setattr(bench, "REF_BUDGET_S", 1e9)
    bench.bench_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == bench.UNIT
    assert "first 3 of the 3 requests" in line["cpu_baseline"]["sample"]
    assert line["e2e"]["value"] == line["value"] > 0
    monkeypatch.setattr(bench, "REF_BUDGET_S", 1e-9)
    bench.bench_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert "first 1 of the 3 requests" in line["cpu_baseline"]["sample"]
    assert line["value"] > 0


def test_code_only_drops_comments_and_layout():
    a = "int f(int x) {  // doubles\n    return 2 * x; /* fast\n path */ }\n"
    b = "int f(int x) {\n return 2 * x; }"
    assert bench._code_only(a) == bench._code_only(b) == "int f(int x) { return 2 * x; }"
    assert bench._code_only(a) != bench._code_only(a.replace("2 * x", "3 * x"))


def _ref_and_gpu():
    rng = np.random.default_rng(3)
    B, N = 6, 5
    ref = {"accept_len": np.array([0, 1, 2, 0, 3, 1], np.int32),
           "out_tokens": rng.integers(0, 100, (B, N)).astype(np.int32),
           "kv_commit": rng.integers(0, N, (B, N)).astype(np.int32),
           "bonus": rng.integers(0, 100, B).astype(np.int32),
           "status": np.zeros(B, np.int32),
           "decision_margin": np.full(B, 1.0), "cdf_margin": np.full(B, 1.0)}
    for b in range(B):
        ref["out_tokens"][b, ref["accept_len"][b]] = ref["bonus"][b]
    ref["cdf_lo"], ref["cdf_hi"] = ref["bonus"] - 1, ref["bonus"] + 1
    gpu = {k: ref[k].copy() for k in bench.OUT_KEYS}
    return ref, gpu


def test_parity_summary_counts():
    ref, gpu = _ref_and_gpu()
    s = bench.parity_summary(gpu, ref)
    assert (s["requests"], s["identical"], s["mismatched"]) == (6, 6, 0)
    # request 1: bonus one token off, near a CDF boundary and inside the window
    ref["cdf_margin"][1] = 1e-8
    L = ref["accept_len"][1]
    gpu["bonus"][1] += 1
    gpu["out_tokens"][1, L] += 1
    # request 2: an accept decision within the margin, decided the other way
    ref["decision_margin"][2] = 1e-9
    gpu["accept_len"][2] -= 1
    # request 3: a plain mismatch
    gpu["kv_commit"][3, 0] += 1
    # request 4: near a boundary but drawn outside the window
    ref["cdf_margin"][4] = 1e-8
    gpu["bonus"][4] += 5
    gpu["out_tokens"][4, ref["accept_len"][4]] += 5
    s = bench.parity_summary(gpu, ref)
    assert s["identical"] == 2                      # requests 0 and 5
    assert s["near_boundary_in_window"] == 1        # request 1
    assert (s["decision_margin_cases"], s["decision_margin_differing"]) == (1, 1)
    assert s["mismatched"] == 2                     # requests 3 and 4


def test_parity_summary_on_the_oracle_outputs():
    """The CPU-baseline leg's oracle outputs carry every field the summary reads."""
    w = W.WORKLOADS["sampling_trie"].scaled(B=3, N=8, V=300, boost=12.0, seed=7)
    x = W.make(w, seed=7)
    value, reps, el, ref = bench.run_oracle_sample(x, w, 2, reps_target_s=0.0, max_reps=1)
    assert reps == 1 and value > 0
    gpu = {k: np.array(ref[k]) for k in bench.OUT_KEYS}
    s = bench.parity_summary(gpu, ref)
    assert s["requests"] == 3 and s["identical"] == 3 and s["mismatched"] == 0

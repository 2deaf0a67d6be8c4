"""Host logic of bench.py that feeds its JSON line (no GPU): clock-sample
summaries, the DRAM-traffic record tied to the kernel's source, the peaks."""
import json
import os

import bench
import synth


def _sampler_with(tmp_path, monkeypatch, rows):
    monkeypatch.setenv("KDA_BENCH_CLOCKS_DIR", str(tmp_path))
    s = bench.ClockSampler(0)
    with open(s.path, "w") as f:
        f.write("\n".join(rows) + "\n")
    s.proc = object()   # stands for a sampler that ran
    return s


def test_clock_summary_loaded_samples_and_reasons(tmp_path, monkeypatch):
    idle = "0, 1200, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    busy = "0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    capped = "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active"
    s = _sampler_with(tmp_path, monkeypatch, [idle, busy, busy, capped, "garbage line"])
    out = s.summary()
    # the idle sample (power under 20 % of the peak) is not "under load"
    assert out["samples"] == 4 and out["samples_under_load"] == 3
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_thermal_slowdown(tmp_path, monkeypatch):
    row = "0, 1500, 2070, 1000.0, 0x40, Not Active, Not Active, Active, Not Active"
    out = _sampler_with(tmp_path, monkeypatch, [row]).summary()
    assert out["reasons"] == ["sw_thermal_slowdown"] and out["sm_mhz"] == 1500.0


def test_clock_summary_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("KDA_BENCH_CLOCKS_DIR", str(tmp_path))
    assert bench.ClockSampler(0).summary()["sm_mhz"] is None


def test_traffic_record_follows_the_kernel_source(monkeypatch):
    with open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        rec = json.load(f)["fused_kernel"]
    assert rec["bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
    # the record is reported exactly when it was taken on the source as it stands
    current = rec["source_digest"] == bench.source_digest(*rec["sources"])
    assert bench.ncu_traffic("fused_kernel") == (rec["bytes_per_launch"] if current else None)
    monkeypatch.setattr(bench, "source_digest", lambda *names: rec["source_digest"])
    assert bench.ncu_traffic("fused_kernel") == rec["bytes_per_launch"]
    # a record taken on one workload is not reported for another
    assert bench.ncu_traffic("fused_kernel", rec["workload_name"]) == rec["bytes_per_launch"]
    assert bench.ncu_traffic("fused_kernel", "another_workload") is None
    # any change to the kernel's source voids it
    monkeypatch.setattr(bench, "source_digest", lambda *names: "0" * 16)
    assert bench.ncu_traffic("fused_kernel") is None
    assert bench.ncu_traffic("no_such_kernel") is None


def test_peaks_fall_back_when_unmeasured(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (6800.0, 1900.0, "of fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000, "bf16_tflops": 2000}))
    assert bench.peaks() == (7000.0, 2000.0, "of measured")


def test_algorithmic_work_per_token_head():
    # 6KV + 2C(3K + 2V) flops and q, k, v, g, out (256 B each) + beta (2 B)
    assert bench.FLOP_PER_TH == 118784
    assert bench.BYTES_PER_TH == 1282


def test_algorithmic_work_counts_state_traffic_per_call():
    import numpy as np
    d = {"q": np.zeros((1, 64, 2, 128), np.uint16), "N": 1,
         "initial_state": np.zeros((1, 2, 128, 128), np.uint16)}
    b1, f1, th = bench.algorithmic_work(d, 1)
    assert th == 128 and f1 == bench.FLOP_PER_TH * 128
    assert b1 == bench.BYTES_PER_TH * 128 + 2 * 128 * 128 * (2 + 4)
    # two calls carrying an fp32 state: the second reads 4 B per element, both write 4 B
    d["initial_state"] = None
    b2, _, _ = bench.algorithmic_work(d, 2)
    assert b2 == bench.BYTES_PER_TH * 128 + 2 * 128 * 128 * ((0 + 4) + (4 + 4))


def test_cpu_baseline_one_thread_figure():
    """Fixed-length workloads of at least 1,024 tokens carry a one-thread oracle figure
    (the first 1,024 tokens of head 0, extrapolated); varlen ones do not."""
    d = synth.make_inputs(1, 1024, 2, seed=0, init_dtype="bf16")
    rec = bench.cpu_baseline(d, "fixed", target_s=0.1)
    assert rec["kind"] == "oracle" and rec["value"] > 0
    one = rec["one_thread"]
    assert one["cores"] == 1 and one["value"] > 0 and "first 1024 tokens" in one["sample"]
    dv = synth.make_inputs(1, 1100, 1, seed=0, lengths=[600, 500])
    assert "one_thread" not in bench.cpu_baseline(dv, "varlen", target_s=0.1)

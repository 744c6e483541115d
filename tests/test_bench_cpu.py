"""Host-side bookkeeping of bench.py (CPU only): the clock record taken during the
timed region, the ncu traffic lookup keyed by the kernel sources' hash, the peak
denominators and the oracle sample behind the GroupedMatMul CPU baseline."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

NA = "Not Active"


def _row(uuid, sm, mx, hw=NA, hw_th=NA, sw_th=NA, cap=NA, index=0):
    return f"{index}, {uuid}, {sm}, {mx}, 700.00, 0x0, {hw}, {hw_th}, {sw_th}, {cap}"


def _summary(tmp_path, lines, uuid="GPU-a"):
    path = tmp_path / "clocks.csv"
    path.write_text("\n".join(lines) + "\n")
    s = bench.ClockSampler(uuid)
    s.out = open(path)          # summary() reads the file by name and removes it
    s.out.close()
    s.proc = object()           # samples were taken
    return s.summary()


def test_clock_median_under_load_ignores_idle_samples(tmp_path):
    rows = [_row("GPU-a", 345, 2070)] + [_row("GPU-a", 2070, 2070)] * 5 + [_row("GPU-a", 1980, 2070)]
    got = _summary(tmp_path, rows)
    assert got["sm_mhz"] == 2070 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == [] and got["samples"] == 7


def test_clock_reasons_are_collected(tmp_path):
    rows = [_row("GPU-a", 2070, 2070, cap="Active"), _row("GPU-a", 1500, 2070, hw_th="Active"),
            _row("GPU-a", 2070, 2070)]
    got = _summary(tmp_path, rows)
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_clock_rows_of_other_gpus_are_dropped(tmp_path):
    rows = [_row("GPU-a", 2070, 2070), _row("GPU-b", 900, 2070, hw="Active", index=1)]
    got = _summary(tmp_path, rows)
    assert got["samples"] == 1 and got["reasons"] == [] and got["sm_mhz"] == 2070


def test_clock_without_samples(tmp_path):
    assert _summary(tmp_path, [])["reasons"] == ["no samples"]
    s = bench.ClockSampler(None)
    assert s.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_traffic_follows_the_kernel_source_hash(tmp_path, monkeypatch):
    csrc = tmp_path / "quantized_mixture_experts_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("// kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha(["k.cu"])
    (tmp_path / "profiles" / "k_w.md").write_text(
        f"text\n\n    dram_bytes_per_launch: 123456\n    source_sha: {sha}\n")
    assert bench.ncu_traffic("k_w.md", ["k.cu"]) == 123456.0
    assert bench.ncu_traffic("missing.md", ["k.cu"]) is None
    (csrc / "k.cu").write_text("// kernel v2\n")      # the counters no longer describe it
    assert bench.ncu_traffic("k_w.md", ["k.cu"]) is None


def test_profile_blocks_parse():
    """Every summary that carries a machine-readable block gives a byte count and a
    16-hex-digit source hash (bench.py reports null traffic once the hash is stale)."""
    import re
    pdir = os.path.join(ROOT, "profiles")
    seen = 0
    for name in sorted(os.listdir(pdir)):
        text = open(os.path.join(pdir, name)).read()
        if "dram_bytes_per_launch" not in text:
            continue
        seen += 1
        m = re.search(r"dram_bytes_per_launch:\s*([0-9]+)\s*\n\s*source_sha:\s*([0-9a-f]{16})\s*$",
                      text)
        assert m and int(m.group(1)) > 0, name
    assert seen >= 5


def test_peaks_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.measured_peaks()
    assert fb["source"] == "fallback" and (fb["hbm_gbs"], fb["bf16_tflops"]) == (6800.0, 1900.0)
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6772.0, "bf16_tflops": 1936.6, "bf16_tflops_sustained": 1700.0}))
    got = bench.measured_peaks()
    assert got["source"] == "measured" and got["hbm_gbs"] == 6772.0


def test_gmm_oracle_sample_scales_by_the_column_fraction():
    pytest.importorskip("torch")
    from quantized_mixture_experts_gb300.workloads import GMM_WORKLOADS, make_gmm_inputs
    wl = GMM_WORKLOADS["gmm_tiny"]
    dt, rows_eq, what = bench.gmm_oracle_sample(make_gmm_inputs(wl), wl, seed=0, rows=40, cols=50)
    assert dt > 0 and rows_eq == pytest.approx(40 * 50 / wl.N)
    assert what == f"40 of {wl.M} rows x 50 of {wl.N} columns"

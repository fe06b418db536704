"""Host-side logic of bench.py (no GPU): the roofline model of a part, the
nvidia-smi clock summary and its throttle reasons, and the peaks file."""
import json

import numpy as np
import pytest

import bench
import oracle
import spmm_workloads as W


def test_part_model_matches_the_definitions_on_bcsr_tiny():
    """FLOPs: 2*nnz*N (effective) and 2*stored*N (roofline); bytes: stored
    values + format indices + B once + C once."""
    w = W.bcsr_tiny()
    ptr, idx, vals = oracle.bcsr_build(w.m, w.k, w.row_ptr, w.col_idx, w.vals, 64, 64)
    stored = vals.size
    info = {"stored": stored, "idx_bytes": ptr.size * 8 + idx.size * 4}
    eff, stored_fl, bytes_min = bench.part_model(w, info)
    assert eff == 2.0 * w.nnz * w.n
    assert stored_fl == 2.0 * stored * w.n
    out_sz = 4 if w.out_dtype == "f32" else 2
    assert bytes_min == 2 * stored + info["idx_bytes"] + 2 * w.k * w.n + out_sz * w.m * w.n
    # bcsr_tiny keeps whole 64x64 blocks, so stored = nnz
    assert stored == w.nnz


def _sample(sm, mx, **active):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if active.get(n) else "Not Active" for n in names]
    return ", ".join(["0", str(sm), str(mx), "900.0", "0x0"] + flags)


def test_clock_summary_median_under_load_and_reasons():
    c = bench.ClockSampler(0)
    c.lines = [_sample(345, 2070), _sample(2070, 2070), _sample(2040, 2070, sw_power_cap=True),
               _sample(2070, 2070), _sample(1995, 2070, hw_slowdown=True), "garbage line"]
    s = c.summary()
    assert s["samples"] == 5
    assert s["sm_max_mhz"] == 2070.0
    # the idle sample (345 MHz, below half the maximum) is left out of the median
    assert s["sm_mhz"] == float(np.median([2070, 2040, 2070, 1995]))
    assert s["reasons"] == ["hw_slowdown", "sw_power_cap"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler(0).summary()
    assert s["sm_mhz"] is None and s["samples"] == 0 and s["reasons"] == []


def test_peaks_file_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.load_peaks()
    assert fb["source"] == "fallback" and fb["hbm_gbs"] == 6800.0 and fb["bf16_tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 1.5, "bf16_tflops": 2.5}))
    pk = bench.load_peaks()
    assert pk == {"hbm_gbs": 1.5, "bf16_tflops": 2.5, "bf16_tflops_sustained": None, "source": "measured"}


def test_traffic_key_ignores_comments_only(tmp_path, monkeypatch):
    csrc = tmp_path / "sparse_dense_matrix_bcsr_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (csrc / "k.cu").write_text("int a = 1;  // one\n\nint b = 2;\n")
    h0 = bench.src_sha("k.cu")
    (csrc / "k.cu").write_text("// header\nint a = 1;\nint b = 2;  // two\n")
    assert bench.src_sha("k.cu") == h0
    (csrc / "k.cu").write_text("int a = 1;\nint b = 3;\n")
    assert bench.src_sha("k.cu") != h0


def test_gather_model_counts_one_b_row_per_packed_column():
    class _W:  # the two fields gather_model reads
        fmt, n = "wcsr", 256
    assert bench.gather_model(_W, {"n_units": 1000}) == 2.0 * 1000 * 256
    _W.fmt = "bcsr"
    assert bench.gather_model(_W, {"n_units": 1000}) == 0.0


@pytest.mark.parametrize("entry,base,flags,point", [
    ("wcsr_uniform", "wcsr_uniform", {}, None),
    ("wcsr_irregular_rcm_dyn", "wcsr_irregular", {"rcm": True, "dyn": True}, None),
    ("wcsr_uniform_h64", "wcsr_uniform", {"h64": True}, None),
    ("bcsr_sweep_95_N256_split", "bcsr_sweep_95_N256", {"split": True}, ("bcsr", 95.0, 256)),
    ("wcsr_sweep_0.1_N8_h64", "wcsr_sweep_0.1_N8", {"h64": True}, ("wcsr", 0.1, 8)),
    ("wcsr_sweep_2.0_N256_rcm", "wcsr_sweep_2.0_N256", {"rcm": True}, ("wcsr", 2.0, 256)),
])
def test_sweep_entry_parsing(entry, base, flags, point):
    b, f, pt = bench.parse_config_entry(entry)
    assert (b, f, pt) == (base, flags, point)

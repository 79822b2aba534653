"""bench.py's rate and roofline arithmetic (CPU only, on made-up kernel timings).

The bench line's fractions are the judged numbers, so the choice of peak is
checked here: the burst bf16 rate for a timed region under two seconds, the
sustained one for a longer region, the UMMA rate at the sampled clock beside
them; the fp32 path (CUDA cores) against the fp32 FMA rate; and byte-bound
kernels against the measured copy bandwidth.
"""
import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PEAKS = {"bf16_tflops": 1854.8, "bf16_tflops_sustained": 1699.2, "hbm_gbs": 6784.5}


@pytest.fixture(scope="module")
def bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    mod.sm_count = lambda: 152
    return mod


def result(kernels, steps=20, timed_s=0.45, mhz=2000.0, ds_bytes=0):
    return {"steps": steps, "clocks": {"sm_mhz": mhz} if mhz else None, "timed_s": timed_s,
            "ds_bytes": ds_bytes, "kernels": kernels, "s2h_qkv_ms": 0.1, "h2s_o_ms": 0.1, "fwd_ms": 1.0,
            "bwd_ms": 2.0, "ms_per_step": 3.0, "path": "fused"}


def test_short_bf16_region_is_held_to_the_burst_peak(bench):
    w = bench.WORKLOADS["llama8b_8k"]
    fl = bench.attn_flops(w, offs=bench.doc_offsets_for(w))
    ms = 0.5
    rs = bench.run_summary(w, result({"attn_fwd": {"total_ms": 20 * ms, "launches": 20, "ms_per_step": ms}}),
                           PEAKS, "measured")
    roof = rs["roofline"]
    achieved = fl / (ms * 1e-3) / 1e12
    assert roof["bound"] == "tensor" and roof["peak"] == PEAKS["bf16_tflops"]
    assert roof["achieved"] == pytest.approx(achieved)
    assert roof["frac"] == pytest.approx(achieved / PEAKS["bf16_tflops"])
    assert roof["frac_sustained"] == pytest.approx(achieved / PEAKS["bf16_tflops_sustained"])
    # 8192 flop/cycle/SM x 152 SMs x 2000 MHz
    assert roof["frac_of_clock_peak"] == pytest.approx(achieved / (8192 * 152 * 2000e6 / 1e12))


def test_long_bf16_region_is_held_to_the_sustained_peak(bench):
    w = bench.WORKLOADS["llama8b_8k"]
    rs = bench.run_summary(w, result({"attn_fwd": {"total_ms": 10.0, "launches": 20, "ms_per_step": 0.5}},
                                     timed_s=3.0), PEAKS, "measured")
    assert rs["roofline"]["peak"] == PEAKS["bf16_tflops_sustained"]
    assert "sustained" in rs["roofline"]["peak_source"]


def test_fp32_path_is_alu_bound_against_the_fp32_fma_rate(bench):
    w = bench.WORKLOADS["tiny"]
    fl = bench.attn_flops(w, offs=bench.doc_offsets_for(w))
    ms = 0.1
    # too short for a clock sample: the maximum SM clock stands in
    rs = bench.run_summary(w, result({"attn_fwd": {"total_ms": 20 * ms, "launches": 20, "ms_per_step": ms}},
                                     timed_s=0.002, mhz=None), PEAKS, "measured")
    roof = rs["roofline"]
    peak = 256 * 152 * 2070e6 / 1e12
    assert roof["bound"] == "alu" and roof["peak"] == pytest.approx(peak)
    assert roof["frac"] == pytest.approx(fl / (ms * 1e-3) / 1e12 / peak)
    assert "frac_burst" not in roof and "maximum SM clock" in roof["peak_source"]
    assert rs["kernels"]["attn_fwd"]["bound"] == "alu"
    assert "frac_burst" not in rs["kernels"]["attn_fwd"]


def test_stored_ds_dq_kernel_is_counted_in_bytes(bench):
    w = bench.WORKLOADS["llama8b_32k"]
    blocks = 4 << 30
    kernels = {"attn_fwd": {"total_ms": 100.0, "launches": 20, "ms_per_step": 5.0},
               "bwd_dq": {"total_ms": 80.0, "launches": 20, "ms_per_step": 4.0}}
    rs = bench.run_summary(w, result(kernels, ds_bytes=blocks + 32768), PEAKS, "measured")
    dq = rs["kernels"]["bwd_dq"]
    assert "gbs" in dq and "tflops" not in dq
    assert dq["frac_hbm"] == pytest.approx(dq["gbs"] / PEAKS["hbm_gbs"])
    # the forward has the larger share of the step here: the roofline is its
    assert rs["roofline"]["kernel"] == "attn_fwd_sm103_kernel"

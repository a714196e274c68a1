"""Host-side logic of bench.py on the CPU: the roofline of a workload, the
clock summary of the nvidia-smi samples, and the recorded DRAM traffic that
is reported only for the kernel sources it was captured on."""

import bench
from transformer_linear_layer_tcgen05_gb300 import workloads as wl

PEAKS = {"hbm_gbs": 6784.5, "bf16_tflops": 1878.3, "bf16_tflops_sustained": 1704.2}


def test_roofline_bounds():
    head = wl.WORKLOADS_BY_NAME["ffn_down_swiglu_w16_16k"]
    bound, roof, tpeak, hbm = bench.roofline(head, PEAKS)
    assert bound == "tensor" and roof == tpeak == 1878.3 and hbm == 6784.5
    assert bench.roofline(head, PEAKS, sustained=True)[1] == 1704.2
    small = wl.WORKLOADS_BY_NAME["attn_proj_f32"]
    bound, roof, tpeak, _ = bench.roofline(small, PEAKS)
    # TF32 at the nominal ratio of the bf16 peak; HBM-bound: FLOPs / bytes x bandwidth
    assert bound == "hbm" and tpeak < 1878.3
    nbytes = wl.input_bytes(small.form, small.M, small.N, small.K)
    assert abs(roof - small.flops / nbytes * 6784.5 / 1e3) < 1e-6


def _sampler(rows):
    s = bench.ClockSampler(None)
    s.samples = rows
    return s


def test_clock_summary_median_reasons_and_window():
    row = lambda mhz, power, slow="Not Active", cap="Not Active": [
        "ts", str(mhz), "2070", str(power), "0x0", slow, "Not Active", "Not Active", cap]
    s = _sampler([(0.5, row(2070, 300)),                          # before the region
                  (1.0, row(1900, 1390, cap="Active")),
                  (1.2, row(1800, 1395, cap="Active")),
                  (1.4, row(1700, 1380, cap="Active")),
                  (5.0, row(600, 100, slow="Active"))])           # after it
    out = s.summary(1.0, 1.5)
    assert out["sm_mhz"] == 1800 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 1395 and out["samples_in_timed_region"] == 3
    out = s.summary(4.9, 5.0)
    assert out["reasons"] == ["hw_slowdown"]


def test_clock_summary_without_samples():
    out = _sampler([]).summary(0.0, 1.0)
    assert out["samples"] == 0 and out["sm_mhz"] is None


def test_recorded_traffic_needs_the_captured_sources(monkeypatch):
    got = bench.recorded_traffic("ffn_down_swiglu_w16_16k")
    if got is not None:   # recorded for the current sources: a positive byte count
        assert got > 0
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0000000000000000")
    assert bench.recorded_traffic("ffn_down_swiglu_w16_16k") is None
    assert bench.recorded_traffic("no_such_workload") is None

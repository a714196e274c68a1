"""Host-side logic of bench.py on the CPU: the roofline of a workload, the
clock summary of the nvidia-smi samples, and the recorded DRAM traffic that
is reported only for the kernel sources it was captured on."""

import os

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
    smi = lambda t, mhz, power, slow="Not Active", cap="Not Active": \
        bench.ClockSampler.parse_smi_row(
            t, f"ts, {mhz}, 2070, {power}, 0x0, {slow}, Not Active, Not Active, {cap}")
    s = _sampler([smi(0.5, 2070, 300),                             # before the region
                  smi(1.0, 1900, 1390, cap="Active"),
                  smi(1.2, 1800, 1395, cap="Active"),
                  smi(1.4, 1700, 1380, cap="Active"),
                  smi(5.0, 600, 100, slow="Active")])              # after it
    out = s.summary(1.0, 1.5)
    assert out["sm_mhz"] == 1800 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 1395 and out["samples_in_timed_region"] == 3
    out = s.summary(4.9, 5.0)
    assert out["reasons"] == ["hw_slowdown"]
    # NVML-style samples (the in-process sampler's own tuples) read the same way
    s = _sampler([(1.000, 2070.0, 2070.0, 900.0, frozenset()),
                  (1.002, 2055.0, 2070.0, 950.0, frozenset({"sw_power_cap"})),
                  (1.004, 2040.0, 2070.0, 940.0, frozenset())])
    out = s.summary(1.0, 1.011)
    assert out["samples_in_timed_region"] == 3 and out["sm_mhz"] == 2055.0
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_without_samples():
    out = _sampler([]).summary(0.0, 1.0)
    assert out["samples"] == 0 and out["sm_mhz"] is None


def test_tf32_peak_is_the_recorded_one_when_present():
    peaks = dict(PEAKS, tf32_tflops=1000.0, tf32_tflops_sustained=900.0)
    assert bench.tensor_peak("tf32", peaks)[0] == 1000.0
    assert bench.tensor_peak("tf32", peaks, sustained=True)[0] == 900.0
    assert bench.tensor_peak("f16", peaks)[0] == 1878.3      # f16: the bf16 measurement
    # without a recorded TF32 figure: the nominal ratio of the bf16 peak
    assert abs(bench.tensor_peak("tf32", PEAKS)[0] - 1878.3 * 1.1 / 2.25) < 1e-9
    dx = wl.WORKLOADS_BY_NAME["ffn_up_dx_f32"] if "ffn_up_dx_f32" in wl.WORKLOADS_BY_NAME \
        else [b for b in wl.BACKWARD_WORKLOADS if b.name == "ffn_up_dx_f32"][0]
    assert bench.roofline(dx, dict(PEAKS, tf32_tflops=50.0))[0] == "tensor"
    rec = bench.recorded_tensor_peaks()
    assert all(k in ("tf32_tflops", "tf32_tflops_sustained") and v > 0 for k, v in rec.items())


def test_launch_command_reruns_this_script_as_ranks():
    cmd = bench.launch_command(4, ["--gpus", "4", "--steps", "20"], 29555)
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=4" in cmd and cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[cmd.index("--master-port") + 1] == "29555"
    assert os.path.samefile(cmd[-5], bench.__file__)
    assert cmd[-4:] == ["--gpus", "4", "--steps", "20"]


def test_recorded_traffic_needs_the_captured_sources(monkeypatch):
    got = bench.recorded_traffic("ffn_down_swiglu_w16_16k")
    if got is not None:   # recorded for the current sources: a positive byte count
        assert got > 0
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0000000000000000")
    assert bench.recorded_traffic("ffn_down_swiglu_w16_16k") is None
    assert bench.recorded_traffic("no_such_workload") is None

"""Host-side logic of bench.py (no GPU): the algorithmic FLOPs and bytes that
the roofline fractions divide by, checked against the layer's shapes worked
out by hand; the roofline entry's choice of bound and peak; the clock
summary's decoding of NVML clock-event reasons (with a fake reader)."""
import math

import pytest

import bench
import moe_inputs


def test_prefill_gate_up_and_down_work():
    # Mixtral-shaped prefill: 8192 kept assignments, all 8 experts active
    w = moe_inputs.WORKLOADS["mixtral_prefill"]
    work = bench.algorithmic_work(w, 8192, 8)
    gu_f, gu_b = work["gate_up"]
    dn_f, dn_b = work["down"]
    assert gu_f == 2 * 8192 * 4096 * (2 * 14336)                   # 1.924 TFLOP
    assert gu_b == 8 * 2 * 14336 * 4096 * 2 + 8192 * 4096 * 2 + 8192 * 14336 * 2
    assert gu_b == 2181038080
    assert dn_f == 2 * 8192 * 14336 * 4096
    assert dn_b == 8 * 14336 * 4096 * 2 + 8192 * 14336 * 2 + 8192 * 4096 * 4
    lf, lb = work["layer"]
    assert lf == gu_f + dn_f == 6 * 8192 * 4096 * 14336
    # every active expert's three matrices once, x in, y out, the fp32 router
    assert lb == 8 * 3 * 14336 * 4096 * 2 + 2 * 4096 * 4096 * 2 + 8 * 4096 * 4


def test_inactive_experts_cost_no_weight_bytes():
    w = moe_inputs.WORKLOADS["switch_skewed"]
    a = bench.algorithmic_work(w, 12316, 64)["gate_up"][1]
    b = bench.algorithmic_work(w, 12316, 32)["gate_up"][1]
    assert a - b == 32 * 2 * w.F * w.d * 2


def test_switch_down_with_the_combine_fused():
    # K = 1, no shared experts: the down projection writes the kept tokens' y
    # (bf16) and reads their residual rows instead of writing fp32 o
    w = moe_inputs.WORKLOADS["switch_skewed"]
    assert bench.combine_fused(w)
    dn_b = bench.algorithmic_work(w, 12316, 64)["down"][1]
    assert dn_b == 64 * 1024 * 4096 * 2 + 12316 * 4096 * 2 + 12316 * 1024 * 2 * 2
    assert not bench.combine_fused(moe_inputs.WORKLOADS["mixtral_prefill"])   # K = 2
    assert not bench.combine_fused(moe_inputs.WORKLOADS["tiny_fp32"])         # CUDA cores


def test_backward_work_is_twice_the_forward_flops():
    w = moe_inputs.WORKLOADS["mixtral_prefill"]
    bw = bench.backward_work(w, 8192, 8)
    fw = bench.algorithmic_work(w, 8192, 8)
    bwd_flops = sum(bw[k][0] for k in ("bwd_down_dgrad", "bwd_down_wgrad",
                                        "bwd_gate_up_dgrad", "bwd_gate_up_wgrad"))
    assert bwd_flops == 2 * fw["layer"][0]
    assert bw["step"][0] == 3 * fw["layer"][0]
    # the weight-gradient launches write every expert's fp32 gradients
    E, d, F = w.N, w.d, w.F
    assert bw["bwd_gate_up_wgrad"][1] >= E * 2 * F * d * 4
    assert bw["bwd_down_wgrad"][1] >= E * d * F * 4


PEAKS = {"hbm_gbs": 6500.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def test_roofline_picks_the_larger_roofline_time():
    # 1.8 TFLOP and 1 GB: 1 ms on the tensor cores, 0.15 ms of HBM -> tensor
    r = bench.roofline_entry(1.8e12, 1e9, 2e-3, PEAKS)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert math.isclose(r["achieved"], 900.0) and math.isclose(r["frac"], 0.5)
    # 1 GFLOP and 6.5 GB: HBM-bound
    r = bench.roofline_entry(1e9, 6.5e9, 2e-3, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert math.isclose(r["achieved"], 3250.0) and math.isclose(r["frac"], 0.5)


def test_roofline_sustained_peak_when_power_capped():
    r = bench.roofline_entry(1.4e12, 1e9, 1e-3, PEAKS, sustained=True)
    assert r["peak"] == 1400.0 and math.isclose(r["frac"], 1.0)
    r = bench.roofline_entry(1.4e12, 1e9, 1e-3, PEAKS, sustained=False)
    assert r["peak"] == 1800.0 and r["frac"] == pytest.approx(1400 / 1800, abs=1e-4)


class _FakeNvml:
    """Stands in for the NVML reader: a clock trace and reason bits."""

    def __init__(self):
        self.mhz = iter([2032, 1995, 1260, 1250, 1255] + [1255] * 1000)
        self.bits = iter([0x1, 0x4, 0x4 | 0x8] + [0x4] * 1000)

    def sm_max_mhz(self):
        return 2032

    def sm_mhz(self):
        return next(self.mhz)

    def reasons(self):
        return next(self.bits)


def test_clock_summary_decodes_reasons(monkeypatch):
    monkeypatch.setattr(bench, "_NvmlReader", _FakeNvml)
    cs = bench.ClockSampler(period_s=0.0)
    for _ in range(5):  # the sampling thread's work, done inline
        cs.samples.append(cs.nvml.sm_mhz())
        cs.reason_bits |= cs.nvml.reasons()
    s = cs.summary()
    assert s["sm_max_mhz"] == 2032 and s["samples"] == 5
    assert s["sm_mhz"] == 1260                       # median of the five samples
    assert s["reasons"] == ["sw_power_cap", "hw_slowdown"]   # gpu_idle is not reported


def test_clock_summary_without_nvml(monkeypatch):
    def broken():
        raise RuntimeError("no device")
    monkeypatch.setattr(bench, "_NvmlReader", broken)
    with bench.ClockSampler() as cs:
        pass
    s = cs.summary()
    assert s["sm_mhz"] is None and s["reasons"] == [] and "nvml unavailable" in s["note"]


def test_reference_arm_json_line():
    """bench.py --impl reference (the float64 oracle on the host) prints one
    JSON line with the contract's keys; it needs no GPU."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--workload", "mixtral_decode", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["value"] > 0 and j["unit"] == "tokens/s"
    assert j["steps"] == 1 and j["warmup"] == 1 and j["higher_is_better"] is True
    assert j["config"]["workload"] == "mixtral_decode"
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": j["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_ep_staging_bytes():
    # 8192 kept rows leave the source; device 0 of 8 (one expert each)
    # receives 8 * 1000 rows; d = 4096 in bf16, outputs in fp32
    b = bench.ep_bytes(8192, 8000, 4096, 2)
    assert b["ep_pack"] == 2 * 8192 * 4096 * 2
    assert b["ep_unpack"] == 2 * 8192 * 4096 * 4
    assert b["ep_regroup"] == 2 * 8000 * 4096 * 2
    assert b["ep_regroup_back"] == 2 * 8000 * 4096 * 4


def test_measured_traffic_entry():
    # the gate/up GEMM's DRAM bytes from a one-launch ncu capture (read +
    # write), stored with the fingerprint of the kernel sources it was taken
    # on: within 5 % of the launch's algorithmic bytes (no weight tile
    # fetched twice), and the fingerprint well formed and reproducible
    for key, algorithmic in ((("mixtral_prefill", "gate_up"), 2181038080),
                             (("mixtral_prefill", "down"), None)):
        traffic, fp = bench.MEASURED_TRAFFIC[key]
        assert traffic > 0
        if algorithmic is not None:
            assert traffic <= 1.05 * algorithmic
        assert len(fp) == 16 and int(fp, 16) >= 0
    assert bench.kernel_fingerprint() == bench.kernel_fingerprint()

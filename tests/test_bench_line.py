"""The bench line's assembly on CPU: the roofline arithmetic, the clock record
and the keys of the JSON line, with the device queries replaced by fixed
values (no GPU is used)."""
import argparse
import types

import pytest

import bench
import synth

N = 28 * 2 * 8 * 4096 * 128
MED = {"encode": 2.25, "decode": 4.05, "ideal_bits": 1.38}


@pytest.fixture
def fixed_peaks(monkeypatch):
    monkeypatch.setattr(bench, "issue_peak_gops", lambda: (152 * 128 * 2070.0 * 1e6 / 1e9, 152, 2070.0))
    monkeypatch.setattr(bench, "measured_peaks", lambda: (6775.3, "measured"))
    monkeypatch.setattr(bench, "load_traffic", lambda kernel, workload: 1_076_000_000)


def test_roofline_arithmetic(fixed_peaks):
    nb = 168_754_632
    roof, kernels = bench.roofline(MED, N, nb, 2, "qwen3-0.6b-bf16")
    peak = 152 * 128 * 2070.0 * 1e6 / 1e9
    assert roof["kernel"] == "k_decode" and roof["bound"] == "alu" and roof["unit"] == "Gop/s"
    achieved = 180 * N / (4.05e-3) / 1e9
    assert roof["achieved"] == pytest.approx(achieved, rel=1e-4)
    assert roof["frac"] == pytest.approx(achieved / peak, abs=1e-4)
    assert roof["ops_per_scalar"] == 180 and "minimum" in roof["ops_basis"]
    assert "measured" in roof["ops_basis"]
    assert roof["traffic"] == 1_076_000_000
    # HBM view: the container, mu and the decoded cache per scalar
    assert roof["hbm"]["algorithmic_bytes_per_scalar"] == pytest.approx(nb / N + 2 + 2, abs=1e-4)
    assert roof["hbm"]["peak"] == 6775.3
    for op, ms in MED.items():
        ops = bench.ALG_OPS[2][op] * N / (ms * 1e-3) / 1e9
        assert kernels[op]["alu_frac"] == pytest.approx(ops / peak, abs=1e-4)
    # e4m3 and the order-0 baseline take their own per-unit figures
    roof8, _ = bench.roofline(MED, N, nb // 3, 1, "qwen3-8b-e4m3")
    assert roof8["ops_per_scalar"] == 125
    roof0, k0 = bench.roofline(MED, N, nb * 2, 2, "qwen3-0.6b-bf16", order0=True)
    assert roof0["kernel"] == "k_decode_o0" and roof0["ops_per_scalar"] == 90
    assert roof0["hbm"]["algorithmic_bytes_per_scalar"] == pytest.approx(2 * nb / N + 2, abs=1e-4)


def test_clock_record_median_and_reasons():
    c = bench.ClockSampler(0)
    c.lines = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 2055, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
               "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage line"]
    s = c.summary()
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.ClockSampler(0).summary() is None


def test_json_line_keys(fixed_peaks):
    spec = synth.WORKLOADS["qwen3-0.6b-bf16"]
    args = argparse.Namespace(workload=spec.name, steps=30, warmup=3, no_cpu_baseline=True,
                              order0=False, adaptive=False, block_scale=False)
    clk = types.SimpleNamespace(summary=lambda: {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0,
                                                 "reasons": [], "samples": 2})
    e2e = {"value": 40.0, "unit": "GB/s", "h2d_bytes_per_step": 2 * N + 2 * N,
           "d2h_bytes_per_step": 168_754_632 + 2 * N}
    nb, bits = 168_754_632, 5.722 * N
    med = {"encode_with_bits": 3.3, "decode": MED["decode"]}
    alone = {"encode": MED["encode"], "ideal_bits": MED["ideal_bits"]}
    line = bench.finish_line(args, 0, 1, spec, N, nb, bits, 5.70 * N, 2, 7.68,
                             2 * N / 7.68e-3 / 1e9, med, clk, e2e, None, alone=alone,
                             fused_bits=True)
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["metric"] == bench.METRIC and line["unit"] == "GB/s" and line["n_gpus"] == 1
    assert line["higher_is_better"] is True and line["scaling"] == "strong"
    assert line["config"]["workload"] == spec.name
    assert "inside the encoder" in line["config"]["step"]
    # encode (5) + the bits' final sum (1) + bf16 decode (4) per step
    assert line["gpu_launches"] == 10 * 30
    assert line["encode_with_bits_gbs"] == pytest.approx(2 * N / 3.3e-3 / 1e9, abs=0.01)
    assert line["encode_alone_gbs"] == pytest.approx(2 * N / MED["encode"] / 1e6, abs=0.01)
    assert line["roofline"]["kernel"] == "k_decode"          # 4.05 ms > 3.3 ms
    assert line["kernels"]["encode_with_bits"]["kernel"] == "k_encode (ideal bits inside)"
    assert line["kernels_alone"]["ideal_bits"]["kernel"] == "k_ideal"
    # the two passes apart: encode + ideal bits launches as before
    two = bench.finish_line(args, 0, 1, spec, N, nb, bits, 5.70 * N, 2, 7.68, 1.0, med, clk, e2e,
                            None, alone=alone, fused_bits=False)
    assert two["gpu_launches"] == 12 * 30
    assert two["kernels"]["encode_with_bits"]["kernel"] == "k_encode + k_ideal"
    assert line["bits_per_scalar"] == pytest.approx(8.0 * nb / N, abs=1e-5)
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in line["roofline"], k
    nch = 28 * 2 * 8 * 16
    payload = 8.0 * (nb - 64 - 8 * (nch + 1))
    assert line["model_bits_per_scalar"] == pytest.approx(5.70, abs=1e-5)
    assert line["overhead_vs_model_pct"] == pytest.approx(100 * (8.0 * nb / (5.70 * N) - 1), abs=1e-3)
    assert line["payload_overhead_vs_model_pct"] == pytest.approx(
        100 * (payload / (5.70 * N) - 1), abs=1e-3)
    assert bench.finish_line(args, 1, 2, spec, N, nb, bits, None, 2, 7.68, 1.0, med, clk, e2e,
                             None) is None   # only rank 0 prints


def test_cpu_baseline_single_and_all_cores(fixed_peaks):
    """Both oracle legs on the tiny cache: the all-core leg states its cores and
    the CPU model, and codes the same kind of sample as the one-core leg."""
    spec = synth.WORKLOADS["tiny-bf16"]
    w = synth.make(spec)
    n = spec.n
    args = argparse.Namespace(workload=spec.name, steps=3, warmup=3, no_cpu_baseline=False,
                              order0=False, adaptive=False, block_scale=False,
                              cpu_sample_chunks=4)
    clk = types.SimpleNamespace(summary=lambda: None)
    nb, bits = 100_000, 5.2 * n
    line = bench.finish_line(args, 0, 1, spec, n, nb, bits, 5.1 * n, 2, 1.0, 1.0,
                             {"encode": 1.0, "decode": 1.0, "ideal_bits": 1.0}, clk, None, w)
    cpu = line["cpu_baseline"]
    name, cores = bench.host_cpu()
    assert cpu["cores"] == cores >= 1 and cpu["cpu_model"] == name and name
    assert cpu["kind"] == "oracle" and cpu["value"] > 0 and cpu["unit"] == "GB/s"
    assert cpu["single_core"]["cores"] == 1 and cpu["single_core"]["value"] > 0


def test_threaded_oracle_timing_codes_the_same_sample():
    import oracle as O
    spec = synth.WORKLOADS["tiny-bf16"]
    w = synth.make(spec)
    kv, mu, sig, cnt = synth.to_numpy(w)
    m = O.Model(spec.dtype, spec.L, spec.H, spec.T, spec.D, spec.Tb, spec.G, sig, counts=cnt)
    nch = m.num_chunks()
    a = bench.time_oracle(O, m, kv.reshape(-1), mu.reshape(-1), nch, nch)
    b = bench.time_oracle(O, m, kv.reshape(-1), mu.reshape(-1), nch, nch, threads=3)
    assert a[0] == b[0] == spec.n and a[2] == b[2]


def test_size_accounting():
    acc = bench.size_accounting(1000, 1000, 3, 7000.0, 7500.0)
    assert acc["bits_per_scalar"] == 8.0
    assert acc["payload_bits_per_scalar"] == pytest.approx(8.0 * (1000 - 64 - 32) / 1000)
    assert acc["overhead_pct"] == pytest.approx(100 * (8000 / 7000 - 1), abs=1e-3)
    assert acc["overhead_vs_model_pct"] == pytest.approx(100 * (8000 / 7500 - 1), abs=1e-3)

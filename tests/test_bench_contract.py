"""The bench's reference arm (the fp64 oracle on the host cores) prints the
one JSON line the contract asks for; runs on the CPU with the tiny workload."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--config", "0",
                        "--steps", "2", "--warmup", "3"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["config"]["workload"] == "tiny-d64-f256-T256-C64"
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_launch_accounting_matches_the_library():
    """gpu_launches in the bench line counts what the library launches."""
    sys.path.insert(0, ROOT)
    import bench
    from chunk_wise_weight_gb300 import build, ittt
    build.build()
    for B, T, C in ((2, 32768, 2048), (1, 8192, 1024), (1, 256, 256), (1, 1000, 512)):
        assert bench.launches_per_step(B, T, C, None, False) == ittt.launch_count(B, T, 2560,
                                                                                 9728, C)


def test_bench_form_rule_matches_the_library():
    """The bench names the form a call runs from its own copy of the rule
    (the reference arm never loads the CUDA library): it must agree with
    ittt_plan_form."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    from chunk_wise_weight_gb300 import build, ittt
    build.build()
    for B, T, d, f, C in ((8, 2048, 2560, 9728, 512), (4, 4096, 2560, 9728, 1024),
                          (2, 32768, 2560, 9728, 2048), (64, 256, 2560, 9728, 64),
                          (8, 1024, 1024, 3072, 256), (4, 2048, 1024, 3072, 512),
                          (1, 256, 64, 256, 64), (8, 2000, 2560, 9728, 500),
                          (8, 2048, 2560, 9728, 2048), (4, 512, 512, 1024, 128)):
        cfg = dict(B=B, T=T, d=d, f=f, C=C)
        for flags in ({}, {"dual": True}, {"primal": True}, {"l2norm": True},
                      {"fused_conv": True}):
            args = argparse.Namespace(dual=False, primal=False, l2norm=False, fused_conv=False)
            for k, v in flags.items():
                setattr(args, k, v)
            form = ittt.plan_form(B, T, d, f, C, **flags)
            if form < 0:
                continue  # the library rejects the call (e.g. a forced dual form)
            assert bench.dual_form(cfg, args) == (form == ittt.FORM_DUAL), (cfg, flags)


def test_roofline_peak_follows_the_power_state():
    """A tensor-bound kernel is held to the measured sustained peak when the
    timed region's clock record shows the power cap active, else to the
    burst peak (no clock record: burst)."""
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"bf16_tflops": 1925.7, "bf16_tflops_sustained": 1714.9}
    peak, kind = bench.tensor_peak(peaks, "measured", {"reasons": ["sw_power_cap"]})
    assert peak == 1714.9 and "sustained" in kind and "sw_power_cap" in kind
    for clocks in ({"reasons": []}, {"reasons": None}, None, {}):
        peak, kind = bench.tensor_peak(peaks, "measured", clocks)
        assert peak == 1925.7 and "burst" in kind


def test_fp32_input_accounting():
    """fp32 inputs add the four hi/lo split launches per step, triple the
    gate/up and target contractions in the phase model and move 10 bytes per
    split element; the tiny workload runs them by default."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    for B, T, C in ((2, 32768, 2048), (1, 256, 64)):
        assert (bench.launches_per_step(B, T, C, None, False, fp32_inputs=True)
                == bench.launches_per_step(B, T, C, None, False) + 4)
    B, T, d, f, C = 2, 1024, 256, 512, 256
    plain = bench.phase_model(B, T, d, f, C)
    split = bench.phase_model(B, T, d, f, C, fp32_inputs=True)
    assert split["gateup"][1] == 3 * plain["gateup"][1]
    assert split["target"][1] == 3 * plain["target"][1]
    assert split["apply"] == plain["apply"] and split["update"] == plain["update"]
    assert split["conv"][1] == (2 * B * T * d + 2 * f * d + d * d) * 10 + d * 3 * 4
    ns = dict(fp32_inputs=False, bf16_inputs=False, fused_conv=False, shape=None)
    assert bench.fp32_inputs_for(argparse.Namespace(config=0, **ns))
    assert not bench.fp32_inputs_for(argparse.Namespace(config=2, **ns))
    assert not bench.fp32_inputs_for(argparse.Namespace(config=0, **dict(ns, bf16_inputs=True)))
    assert bench.fp32_inputs_for(argparse.Namespace(config=2, **dict(ns, fp32_inputs=True)))

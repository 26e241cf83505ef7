"""bench.py's JSON line: the keys and types every run must print.

The reference arm runs on the CPU (it times the oracle), so its line is checked here without a
GPU; our arm's line is checked on the GPU with a short run.
"""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BASE_KEYS = {"metric": str, "value": (int, float), "unit": str, "n_gpus": int, "steps": int,
             "warmup": int, "ms_per_step": (int, float), "higher_is_better": bool,
             "scaling": str, "dtype": str, "data": str, "config": dict}


def _run(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def _check_base(d):
    for k, t in BASE_KEYS.items():
        assert isinstance(d[k], t), k
    assert "vs_baseline" in d and d["higher_is_better"] is False
    assert d["config"]["workload"]


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--config", "0", "--steps", "1", "--warmup", "0"], 600)
    _check_base(d)
    assert d["impl"] == "reference" and d["dtype"] == "f64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    cb = d["cpu_baseline"]
    assert cb["timed_s"] > 0 and cb["extrapolated"] is False and cb["sampled_flop_fraction"] == 1
    assert d["config"]["config_index"] == 0 and d["config"]["matrices"] == 4


def test_reference_arm_samples_one_iteration_of_the_largest_workload():
    """On the Llama-3-70B share a whole oracle step is about an hour of host time, so each
    reference step runs one 8192x8192 matrix with one Newton–Schulz iteration and says so."""
    import bench
    from workloads import get_config
    wl = get_config(4)
    shapes = [(p.rows, p.cols) for p in wl.params]
    calls = []

    def inputs_of(k):
        calls.append(k)
        r, c = shapes[k]
        return None, None

    import oracle.step as ostep
    orig = ostep.muon_matrix_step
    seen = {}

    def fake(W0, B, cs, **kw):
        seen.update(kw)
        return {}
    ostep.muon_matrix_step = fake
    try:
        spent, flops, what = bench.oracle_muon_sample(wl, shapes, inputs_of, 5.0)
    finally:
        ostep.muon_matrix_step = orig
    assert len(calls) == 1 and shapes[calls[0]] == (8192, 8192)
    assert seen["ns_steps"] == 1
    assert flops == 4 * 8192 ** 3 + 2 * 8192 ** 3
    assert "1 of the 5 Newton–Schulz iterations" in what


@pytest.mark.gpu
def test_our_arm_line():
    d = _run(["--config", "1", "--steps", "3", "--warmup", "3", "--cpu-seconds", "2",
              "--clock-window-s", "0.2"], 900)
    _check_base(d)
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert 0 < r["frac"] < 1.5 and r["achieved"] > 0 and r["peak"] > 0
    assert "traffic" in r
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert e["steps"] == 3  # the same K steps as the device timing
    assert d["gpu_launches"] == 19 * 3
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["device_status"] == 0
    assert d["repack"]["bound"] == "hbm" and d["shampoo"]["bound"] == "tensor"
    assert d["shampoo_tc"]["bound"] == "tensor" and d["shampoo_tc"]["ms"] > 0
    assert d["soap"]["bound"] == "alu" and d["soap"]["ms"] > 0
    assert all(x > 0 for x in d["soap"]["sweeps_per_side"])

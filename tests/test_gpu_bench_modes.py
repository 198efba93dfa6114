"""bench.py on the GPU, on the tiny workload so that each run takes seconds:
every mode the driver or a user runs prints one JSON line with the contract's
keys, a device status of 0 behind it, and (replicas mode) a live parity check
of the timed output against the oracle that passes."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "clocks",
        "e2e", "gpu_launches"}


def _bench(*args):
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "1",
                          "--steps", "3", "--warmup", "3", *args],
                         capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-3000:]
    return json.loads(res.stdout.strip().splitlines()[-1])


def test_default_line_carries_roofline_baseline_and_parity():
    line = _bench("--workload", "tiny", "--cpu-seconds", "1")
    assert KEYS <= set(line) and line["value"] > 0 and line["n_gpus"] == 1
    assert line["roofline"]["frac"] > 0 and line["roofline"]["avg_launch_ms"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["parity"]["pass"] and line["parity"]["rows"] >= 16
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0


@pytest.mark.parametrize("args", [("--qk-norm",), ("--shard", "heads"), ("--shard", "seq"),
                                  ("--proj",)])
def test_other_modes_print_a_line(args):
    line = _bench("--workload", "tiny", "--no-cpu-baseline", *args)
    assert line["value"] > 0 and line["ms_per_step"] > 0 and line["unit"] == "TFLOP/s"

"""bench.py itself: the driver runs it with its own --steps/--warmup, which must not break
any leg of the line.  The GPU test runs the driver's flags on the 7B shape cut to two
layers (the other legs cut likewise); the CPU test runs the reference arm (the oracle) on
the same cut."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _last_json(out: str) -> dict:
    lines = [l for l in out.splitlines() if l.startswith("{")]
    assert lines, out[-2000:]
    return json.loads(lines[-1])


@pytest.mark.gpu
@pytest.mark.parametrize("steps,warmup", [(20, 5), (3, 3)])
def test_bench_with_the_drivers_flags(steps, warmup):
    cmd = [sys.executable, "bench.py", "--steps", str(steps), "--warmup", str(warmup), "--layers", "2",
           "--batched-passes", "2", "--batched-layers", "2", "--long-steps", "2", "--long-layers", "2",
           "--cpu-seconds", "2"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert p.returncode == 0, p.stderr[-3000:]
    line = _last_json(p.stdout)
    assert line["steps"] == steps and line["warmup"] == warmup and line["value"] > 0
    for key in ("roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches", "bitexact"):
        assert line.get(key) is not None, key
    assert line["bitexact"]["equal"] is True and line["bitexact"]["checked_tokens"] >= 2
    assert line["roofline"]["frac"] > 0 and line["e2e"]["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["config"]["first_timed_position"] == 128 + warmup
    assert line["batched_runs"]["value"] > 0 and line["long_context"]["decode"]["value"] > 0


def test_reference_arm_on_the_same_positions():
    """The oracle arm prefills the same prompt and times the same generating positions as
    the GPU arm; its config is the GPU arm's."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--layers", "2", "--steps", "4", "--warmup", "3",
           "--prompt-ids", "6"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-3000:]
    line = _last_json(p.stdout)
    assert line["impl"] == "reference" and line["steps"] == 4 and line["value"] > 0
    assert line["config"]["prompt_ids"] == 6 and line["config"]["first_timed_position"] == 9
    assert "6 prompt ids" in line["config"]["workload"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    import bench

    class Args:
        layers, warmup = 2, 3
    assert bench.workload_config(Args(), 6, 4, "x")["workload"] == line["config"]["workload"]

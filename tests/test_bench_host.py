"""Host logic of bench.py on the CPU: every mode runs to the end and prints one JSON line with its contract's keys.

Each case runs bench.main() in a child process under tests/fake_cuda.py (CUDA calls answered on the host, the
library stubbed), on the named workload shrunk to a few hundred tokens and whole layer groups.  The numbers are
meaningless; what is checked is that each mode gets through the binding's argument checks and assembles its line.
"""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = """
import json, sys
sys.path[:0] = [{tests!r}, {root!r}]
import fake_cuda
fake_cuda.install()
from decode_attention_19_b300 import synth
w = synth.WORKLOADS[{workload!r}]
synth.WORKLOADS[{workload!r}] = w.with_(L=w.G, **{shrink!r})
import bench
sys.argv = ["bench.py"] + {argv!r}
bench.main()
"""

SHRINK = {"llama8b": dict(B=2, T=512), "tiny": dict(B=1, T=64), "evict_quant": dict(B=1, T=4096, T_nominal=16384)}


def run_bench(workload, *argv):
    code = _CHILD.format(tests=os.path.join(ROOT, "tests"), root=ROOT, workload=workload, shrink=SHRINK[workload],
                         argv=["--workload", workload, "--steps", "2", "--warmup", "1", *argv])
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=600,
                       env=dict(os.environ, OMP_NUM_THREADS="2"))
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def _roofline(line):
    roof = line["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in roof, key
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])


@pytest.mark.parametrize("workload,extra", [("llama8b", ["--no-cpu-baseline"]),
                                            ("evict_quant", ["--no-cpu-baseline", "--no-dense"]),
                                            ("tiny", [])])
def test_decode_mode_prints_the_contract_line(workload, extra):
    line = run_bench(workload, *extra)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["config"]["workload"] == workload and line["n_gpus"] == 1 and line["steps"] == 2
    assert line["higher_is_better"] is True and line["scaling"] == "weak"
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step"):
        assert key in line["e2e"], key
    assert line["e2e"]["h2d_bytes_per_step"] > 0 and line["e2e"]["d2h_bytes_per_step"] > 0
    assert line["gpu_launches"] > 0
    assert line["e2e"]["host_us_per_call"] > 0 and line["host_us_per_call"] == line["e2e"]["host_us_per_call"]
    if "--no-dense" not in extra and workload != "tiny":
        assert line["dense_comparator"]["t_call_us"] > 0     # the comparator is timed by default
    _roofline(line)
    if "--no-cpu-baseline" not in extra:
        cb = line["cpu_baseline"]
        assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]


@pytest.mark.parametrize("workload,mode", [("evict_quant", "--evict-plan"), ("llama8b", "--fit-predictor"),
                                           ("llama8b", "--fit-basis")])
def test_write_side_modes_print_their_line(workload, mode):
    line = run_bench(workload, mode)
    for key in ("metric", "value", "unit", "higher_is_better", "config", "roofline"):
        assert key in line, key
    assert line["higher_is_better"] is False and line["config"]["workload"] == workload
    _roofline(line)

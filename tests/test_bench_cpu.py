"""The bench's reference arm (the oracle timed on the host) keeps the JSON-line
contract on the CPU: one line with the contract's keys and the same workload
config as the GPU arm; under torchrun with two ranks only rank 0 prints and both
exit 0."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
        "cpu_baseline", "e2e"}


def _json_lines(out: str):
    return [json.loads(x) for x in out.splitlines() if x.startswith("{")]


def test_workload_config_has_the_same_keys_in_both_arms():
    sys.path.insert(0, ROOT)
    import bench
    from long_context_hybrid_02_b300 import synth
    for w in synth.WORKLOADS.values():
        a = bench.workload_config(w, bench.L2_FLUSHED, bench.GRAPH_TIMING)
        b = bench.workload_config(w, "x", "y")
        assert a.keys() == b.keys()
        assert a["workload"] == w.name and a["ctx"] == w.L and ("Tq" in a) == (not w.decode)
        assert (a["k"] is None) == (w.kind == "hca")


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload",
                        "tiny_csa", "--steps", "1", "--warmup", "0"], cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert KEYS <= d.keys()
    assert d["impl"] == "reference" and d["value"] > 0 and d["n_gpus"] == 1
    assert d["config"]["workload"] == "tiny_csa"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.slow
def test_reference_arm_under_torchrun_prints_on_rank_0_only():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--gpus", "2", "--impl", "reference", "--workload", "tiny_hca", "--steps", "1",
           "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"

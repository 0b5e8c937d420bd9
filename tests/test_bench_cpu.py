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


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_algorithmic_bytes_of_the_64k_csa_step():
    # worked by hand: per row (512 + 128) keys x (K + V) x 512 dims x 2 B, q and o
    # 64 x 512 x 2 B each, 512 int32 indices; per indexer row 16,352 entries x 128
    # x 2 B keys + 16,352 x 4 B scores + 64 x 128 x 2 B q + 64 x 4 B weights
    bench = _bench()
    from long_context_hybrid_02_b300 import synth
    w = synth.WORKLOADS["csa_decode_64k"]
    ne = (w.L - w.n_win) // w.m
    assert ne == 16352
    nb = bench.step_bytes(w, ne, w.n_win)
    assert nb["attention"] == 32 * (640 * 2 * 512 * 2 + 2 * 64 * 512 * 2 + 512 * 4) == 46202880
    assert nb["index"] == 32 * (16352 * 256 + 16352 * 4 + 64 * 256 + 64 * 4) == 136581120
    assert nb["topk"] == 32 * (16352 * 4 + 512 * 4)


def test_traffic_row_applies_only_to_its_workload_kernel_and_source(tmp_path, monkeypatch):
    import hashlib
    bench = _bench()
    src = tmp_path / "long_context_hybrid_02_b300" / "csrc"
    src.mkdir(parents=True)
    (src / "k.cu").write_text("kernel v1\n")
    sha = hashlib.sha256(b"kernel v1\n").hexdigest()[:16]
    (tmp_path / "profiles").mkdir()
    import json
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps({"records": [
        {"workload": "wl_a", "kernel": "attention", "source": "k.cu", "sha256_16": sha,
         "bytes": 12345, "note": "x"}]}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("wl_a", "attention", "k.cu") == 12345.0
    assert bench.profiled_traffic("wl_b", "attention", "k.cu") is None
    assert bench.profiled_traffic("wl_a", "index", "k.cu") is None
    assert bench.profiled_traffic(None, "attention", "k.cu") is None       # not full size
    (src / "k.cu").write_text("kernel v2\n")                                # source changed
    assert bench.profiled_traffic("wl_a", "attention", "k.cu") is None


def test_clock_summary_from_a_fake_nvml(monkeypatch):
    import time
    bench = _bench()
    cs = bench.ClockSampler(None)
    clocks = iter([2032, 1900, 2032, 2032] + [2032] * 10000)
    monkeypatch.setattr(cs, "_open_nvml",
                        lambda: (lambda: next(clocks), lambda: 2032, lambda: 0x4 | 0x1))
    with cs:
        time.sleep(0.05)
    s = cs.summary()
    assert s["sm_mhz"] == 2032 and s["sm_max_mhz"] == 2032 and s["samples"] >= 4
    assert s["reasons"] == ["sw_power_cap"]                # 0x1 (idle) is not reported


def test_clock_summary_names_a_throttle_and_a_missing_nvml(monkeypatch):
    import time
    bench = _bench()
    cs = bench.ClockSampler(None)
    monkeypatch.setattr(cs, "_open_nvml",
                        lambda: (lambda: 1500, lambda: 2032, lambda: 0x8 | 0x40))
    with cs:
        time.sleep(0.02)
    assert cs.summary()["reasons"] == ["hw_slowdown", "hw_thermal_slowdown"]

    def no_nvml():
        raise OSError("libnvidia-ml.so.1: cannot open shared object file")
    cs2 = bench.ClockSampler(None)
    monkeypatch.setattr(cs2, "_open_nvml", no_nvml)
    with cs2:
        pass
    s = cs2.summary()
    assert s["sm_mhz"] is None and s["reasons"][0].startswith("nvml unavailable")

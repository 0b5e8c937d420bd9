#!/usr/bin/env python3
"""Decode throughput of one hybrid-attention layer on B300, printed as one JSON line.

Default workload: CSA decode, 32 sequences at 65,536 tokens, 64 query heads of
dim 512 on one shared K/V head, window 128, m = 4 (16,384 entries per
sequence), top-512, indexer 64 heads x 128, bfloat16 storage, fp32 accumulation.
One step = one decode token per sequence through the whole path, as one call of
the library's fused decode step: compress the block completed by the newest
token (under the disjoint eligibility rule that block is not visible to the step's
own query, so scoring runs beside it), score every eligible entry, select the
top-k, attend to selection + window.  The step's launches are
captured once in a CUDA graph and replayed; timing uses CUDA events recorded at
both ends of the graph on the launching stream, with an L2 flush (256 MiB write,
then 256 MiB read) before every timed step.  The library's kernels are chained
with programmatic dependent launch, so the per-kernel breakdown comes from a
second graph with an event between every two calls.  Other workloads
(--workload): HCA decode at 128K tokens, the million-token decodes, and a CSA
prefill chunk of 4,096 queries (compress the blocks the chunk completes, score,
select, attend; prefill tokens/s).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

With N > 1 (torchrun, one process per GPU) every rank runs its own replica of
the workload (weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the maximum over ranks is reported.
`--impl reference` times the CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="csa_decode_64k")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ctx", type=int, default=0,
                    help="context length (default: the workload's own); a shorter context is a "
                         "smaller workload for profiler captures, not a bench line")
    ap.add_argument("--batch", type=int, default=0,
                    help="sequences (default: the workload's own batch); a smaller batch is a "
                         "smaller workload for profiler captures, not a bench line")
    return ap.parse_args()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and clock-event (throttle) reasons sampled during the timed region.

    Polls the driver's NVML library (read-only queries, through ctypes) from a
    background thread every ~2 ms; the device is found by its PCI bus id, so
    CUDA_VISIBLE_DEVICES remapping does not matter.
    """
    REASONS = {"hw_slowdown": 0x8, "hw_thermal_slowdown": 0x40, "sw_thermal_slowdown": 0x20,
               "sw_power_cap": 0x4, "hw_power_brake_slowdown": 0x80}

    def __init__(self, torch_device):
        self.dev = torch_device
        self.sm, self.reasons, self.smax = [], set(), None
        self.err = None
        self.thread = None

    def _open_nvml(self):
        """The driver's NVML through ctypes: (query functions, device handle)."""
        import ctypes
        import torch
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        pr = torch.cuda.get_device_properties(self.dev)
        bus = f"{pr.pci_domain_id:08x}:{pr.pci_bus_id:02x}:{pr.pci_device_id:02x}.0".encode()
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(h)) != 0:
            raise RuntimeError("device not found by PCI bus id")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        NVML_CLOCK_SM = 1

        def clock(fn):
            v = ctypes.c_uint()
            if fn(h, NVML_CLOCK_SM, ctypes.byref(v)) != 0:
                raise RuntimeError("clock query failed")
            return int(v.value)

        def reasons():
            v = ctypes.c_ulonglong()
            if reasons_fn(h, ctypes.byref(v)) != 0:
                raise RuntimeError("reason query failed")
            return int(v.value)

        return (lambda: clock(lib.nvmlDeviceGetClockInfo),
                lambda: clock(lib.nvmlDeviceGetMaxClockInfo), reasons)

    def __enter__(self):
        import threading
        try:
            sm_clock, max_clock, reasons = self._open_nvml()
            self.smax = max_clock()
        except Exception as e:          # NVML missing: report it, do not guess
            self.err = f"nvml unavailable: {type(e).__name__}: {e}"
            return self
        self.stop = threading.Event()

        def poll():
            while not self.stop.is_set():
                try:
                    self.sm.append(sm_clock())
                    bits = reasons()
                    for name, bit in self.REASONS.items():
                        if bits & bit:
                            self.reasons.add(name)
                except Exception as e:
                    self.err = f"nvml query failed: {e}"
                    return
                time.sleep(0.002)

        self.thread = threading.Thread(target=poll, daemon=True)
        self.thread.start()
        time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.thread is not None:
            self.stop.set()
            self.thread.join(timeout=5)

    def summary(self):
        if not self.sm:
            return {"sm_mhz": None, "sm_max_mhz": self.smax, "reasons": [self.err or "no samples"]}
        return {"sm_mhz": statistics.median(self.sm), "sm_max_mhz": self.smax,
                "reasons": sorted(self.reasons), "samples": len(self.sm), "source": "nvml"}


# ----------------------------------------------------------------------------- helpers
def max_over_ranks(value: float, dev, dist, world: int) -> float:
    """The largest of every rank's `value` (timed milliseconds): the job is as slow as
    its slowest replica."""
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


NOMINAL_HBM_GBS = 7700.0       # B300 HBM3e, nominal
L2_FLUSHED = "flushed before every timed step (256 MiB write, then 256 MiB read)"
GRAPH_TIMING = "CUDA events at both ends of a CUDA graph of the step, per step"


def workload_config(w, l2: str, timing: str) -> dict:
    """The `config` of a JSON line: the workload's sizes (the same keys in both
    arms) and how the line was timed."""
    csa = w.kind == "csa"
    cfg = {"workload": w.name, "kind": w.kind, "B": w.B, "ctx": w.L}
    if not w.decode:
        cfg["Tq"] = w.Tq
    cfg.update({"H": w.H, "d": w.d, "n_win": w.n_win, "m": w.m, "k": w.k if csa else None,
                "H_I": w.H_I if csa else None, "d_I": w.d_I if csa else None,
                "l2": l2, "timing": timing})
    if w.fmt & 2:
        cfg["indexer_format"] = "FP4 keys and queries (e2m1, e4m3 scale per 16), bfloat16 scores"
    if w.fmt & 1:
        cfg["kv_format"] = "compressed K/V: RoPE dims bfloat16, other dims e4m3 + float32 scale per 64"
    return cfg


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


def profiled_traffic(workload: str | None, kernel_name: str, source_file: str):
    """DRAM bytes per launch of `kernel_name` in `workload` from the committed ncu
    table (profiles/dram_traffic.json: a list of {workload, kernel, source, sha256_16,
    bytes, ...} records), or None when there is none or the kernel's source file no
    longer has the SHA-256 prefix it had when the counters were taken."""
    if workload is None:
        return None
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    src = os.path.join(ROOT, "long_context_hybrid_02_b300", "csrc", source_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    for rec in json.load(open(path))["records"]:
        if (rec["workload"] == workload and rec["kernel"] == kernel_name
                and rec["source"] == source_file and rec["sha256_16"] == sha):
            return float(rec["bytes"])
    return None


def step_bytes(w, n_elig: int, n_keys_win: int):
    es = 2 if w.dtype == "bf16" else 4
    row_b = 608 if w.fmt & 1 else w.d * es      # a compressed K or V row
    out = {}
    if w.kind == "csa":
        # FP4 indexer: 80-byte key rows, bfloat16 scores
        key_b = 80 if w.fmt & 2 else w.d_I * es
        score_b = 2 if w.fmt & 2 else 4
        out["compress"] = w.B * (w.m * (2 * w.d + w.d_I) * es + w.m * 4 + 2 * row_b + key_b)
        out["index"] = w.B * (n_elig * key_b + n_elig * score_b + w.H_I * w.d_I * es + w.H_I * 4)
        out["topk"] = w.B * (n_elig * score_b + w.k * 4)
        # FP8 K/V: the selected entries' 608-byte rows (widened in L2), window bf16
        out["attention"] = w.B * (min(w.k, n_elig) * 2 * row_b + n_keys_win * 2 * w.d * es
                                  + 2 * w.H * w.d * es + w.k * 4)
    else:
        out["compress"] = w.B * (w.m * 2 * w.d * es + w.m * 4 + 2 * row_b)
        out["attention"] = w.B * (n_elig * 2 * row_b + n_keys_win * 2 * w.d * es
                                  + 2 * w.H * w.d * es)
    return out


# ----------------------------------------------------------------------------- CPU oracle
def host_buffer_like(t, inputs: bool):
    """Page-locked host staging for the end-to-end copies, from the library's
    ha_host_alloc (write-combined for inputs): host-to-device copies from it
    measured 2.4x faster than from torch's pinned CPU tensors (2 MiB: 46 us
    against 112 us)."""
    from long_context_hybrid_02_b300 import binding as B
    return B.host_empty(tuple(t.shape), t.dtype, write_combined=inputs)


def fp4_indexer_recall(w, tok, qry, layer, dev) -> dict:
    """Diagnostic (untimed, not a gate): share of the bfloat16 indexer's selection
    (bf16 keys, float32 scores) that the FP4 indexer (FP4 keys and queries,
    bfloat16 scores) also selects, on the same tokens and queries, per row, mean
    and minimum."""
    import torch
    from long_context_hybrid_02_b300 import binding as B
    from long_context_hybrid_02_b300.pipeline import HybridLayer
    ref = HybridLayer(w.scaled(fmt=0), tok, dev)
    ref.build_cache()
    out = {}
    for name, lay in (("bf16", ref), ("fp4", layer)):
        B.csa_index_scores(lay.p, qry["qI"], qry["w_idx"], lay.cki, lay.n_cap, qry["q_pos"], 1,
                           lay.scores)
        B.csa_topk(lay.p, lay.scores, lay.n_cap, qry["q_pos"], 1, lay.idx,
                   (lay.ws.data_ptr(), lay.ws.numel()))
        out[name] = lay.idx.reshape(w.B, -1).cpu().numpy()
    torch.cuda.synchronize()
    del ref
    torch.cuda.empty_cache()
    rec = []
    for b in range(w.B):
        a = set(int(i) for i in out["bf16"][b] if i >= 0)
        f = set(int(i) for i in out["fp4"][b] if i >= 0)
        rec.append(len(a & f) / max(1, len(a)))
    return {"mean": round(sum(rec) / len(rec), 4), "min": round(min(rec), 4), "rows": len(rec),
            "against": "bfloat16 indexer keys with float32 scores on the same inputs"}


def bulk_compress_rate(w, layer, dev, reps: int = 3) -> dict:
    """The cache build (every complete block of every sequence compressed in one
    call), timed with CUDA events after an L2 flush: algorithmic bytes = the blocks'
    token rows and gates read plus the compressed rows written."""
    import torch
    n_blk = layer.n_cap
    es = 2 if w.dtype == "bf16" else 4
    rows = (2 * w.d + (w.d_I if w.kind == "csa" else 0)) * es
    rows_out = 2 * (608 if w.fmt & 1 else w.d * es) + \
        ((80 if w.fmt & 2 else w.d_I * es) if w.kind == "csa" else 0)
    nbytes = w.B * n_blk * (w.m * (rows + 4) + rows_out)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = None
    for i in range(reps):
        flush_w.fill_(i)
        torch.cuda.synchronize()
        e0.record()
        layer.build_cache()
        e1.record()
        e1.synchronize()
        ms = e0.elapsed_time(e1)
        best = ms if best is None else min(best, ms)
    del flush_w
    gbs = nbytes / (best * 1e-3) / 1e9
    pk = peaks()
    return {"blocks": w.B * n_blk, "bytes": nbytes, "ms": round(best, 4), "gbs": round(gbs, 1),
            "frac": round(gbs / pk["hbm_gbs"], 4), "timing": f"CUDA events, best of {reps}, "
            "L2 flushed (256 MiB write) before each"}


def oracle_sample(w, tok_host, qry_host, n_seq: int, seconds: float):
    """Run the oracle decode step on sequences of the workload until `seconds` pass.

    Returns (sequences decoded, wall seconds, threads).  The compressed caches of
    the sampled sequences are built by the oracle itself before timing.
    """
    import numpy as np
    import oracle as O

    def f64(t):
        return t.to("cpu").float().numpy().astype(np.float64)

    caches = []
    t = w.L - 1
    ne = O.n_eligible(t, w.n_win, w.m)
    for b in range(n_seq):
        g = tok_host["gate"][b].numpy().astype(np.float64)
        K = f64(tok_host["k_tok"][b])
        V = f64(tok_host["v_tok"][b])
        c = {"K": K, "V": V,
             "ck": O.compress(K, g, w.m, 0, w.n_blocks, w.dtype),
             "cv": O.compress(V, g, w.m, 0, w.n_blocks, w.dtype)}
        if w.kind == "csa":
            c["cki"] = O.compress(f64(tok_host["ki_tok"][b]), g, w.m, 0, w.n_blocks, w.dtype)
        caches.append(c)
    done, t0 = 0, time.perf_counter()
    while True:
        for b, c in enumerate(caches):
            q = f64(qry_host["q"][b, 0])
            if w.kind == "csa":
                O.csa_decode(q, f64(qry_host["qI"][b, 0]), f64(qry_host["w_idx"][b, 0]), c["ck"],
                             c["cv"], c["cki"], c["K"], c["V"], t, n_win=w.n_win, m=w.m, k=w.k,
                             scale=1 / math.sqrt(w.d))
            else:
                O.hca_decode(q, c["ck"], c["cv"], c["K"], c["V"], t, n_win=w.n_win, m=w.m,
                             scale=1 / math.sqrt(w.d))
            done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    el = time.perf_counter() - t0
    return done, el, blas_threads(), ne


def blas_threads() -> int:
    """Threads numpy's BLAS may use (threadpoolctl when present, else the CPU affinity)."""
    try:
        from threadpoolctl import threadpool_info
        return max([d.get("num_threads", 1) for d in threadpool_info()] + [1])
    except ImportError:
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            if os.environ.get(var, "").isdigit():
                return int(os.environ[var])
        return len(os.sched_getaffinity(0))


def host_inputs(w, seqs: int):
    """The workload's inputs for the first `seqs` sequences, drawn on the host."""
    from long_context_hybrid_02_b300 import synth
    ws = w.scaled(B=seqs)
    return synth.make_tokens(ws, "cpu"), synth.make_queries(ws, "cpu")


def scaled_workload(w, args):
    """The workload with the --batch / --ctx overrides applied (both arms)."""
    if args.batch > 0:
        w = w.scaled(B=args.batch)
    if args.ctx > 0:
        w = w.scaled(L=args.ctx)
    return w


def run_reference(args, rank):
    if rank != 0:
        return
    from long_context_hybrid_02_b300 import synth
    w = scaled_workload(synth.WORKLOADS[args.workload], args)
    tok, qry = host_inputs(w, 1)
    per_step = max(0.5, min(5.0, 120.0 / max(1, args.steps + args.warmup)))

    def one(seconds):
        if w.decode:
            d, e, th, _ = oracle_sample(w, tok, qry, 1, seconds)
        else:
            d, e, th = oracle_prefill_sample(w, tok, qry, seconds)
        return d, e, th

    for _ in range(args.warmup):
        one(0.0)
    done, el = 0, 0.0
    for _ in range(args.steps):
        d, e, threads = one(per_step)
        done += d
        el += e
    value = done / el
    cores = len(os.sched_getaffinity(0))
    metric = ("decode tokens/s (one layer, all sequences)" if w.decode
              else "prefill tokens/s (one layer, one chunk)")
    line = {"impl": "reference", "metric": metric,
            "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / max(1, done),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded Gaussian, host-drawn)",
            "config": workload_config(w, "not applicable (host CPU)",
                                      "wall clock of the oracle on the host, per step"),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "host_cpus": cores,
                             "sample": (f"sequence 0 of the workload decoded repeatedly, "
                                        f"{per_step:.1f}s per step" if w.decode else
                                        f"prefill queries of sequence 0, one after the other "
                                        f"from the end of the chunk, {per_step:.1f}s per step")},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- prefill
def oracle_prefill_sample(w, tok_h, qry_h, seconds: float):
    """The oracle's prefill of sequence 0, one query after the other from the end of
    the chunk, until `seconds` pass.  Returns (queries done, wall seconds, threads)."""
    import numpy as np
    import oracle as O

    def f64(t):
        return t.to("cpu").float().numpy().astype(np.float64)

    g = tok_h["gate"][0].numpy().astype(np.float64)
    K, V = f64(tok_h["k_tok"][0]), f64(tok_h["v_tok"][0])
    ck = O.compress(K, g, w.m, 0, w.n_blocks, w.dtype)
    cv = O.compress(V, g, w.m, 0, w.n_blocks, w.dtype)
    cki = O.compress(f64(tok_h["ki_tok"][0]), g, w.m, 0, w.n_blocks, w.dtype)
    done, t0 = 0, time.perf_counter()
    while True:
        i = w.Tq - 1 - (done % w.Tq)
        t = w.L - w.Tq + i
        ne = O.n_eligible(t, w.n_win, w.m)
        sc = O.index_scores(f64(qry_h["qI"][0, i]), f64(qry_h["w_idx"][0, i]), cki[:ne])
        idx = O.topk_select(sc, w.k)
        O.prefill_query(f64(qry_h["q"][0, i]), idx, ck, cv, K, V, t, n_win=w.n_win, m=w.m,
                        scale=1 / math.sqrt(w.d))
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return done, time.perf_counter() - t0, blas_threads()


def run_prefill(args, w, dev, world, rank, dist):
    """One prefill chunk of Tq queries per sequence: compress the blocks the chunk's
    tokens complete, index every eligible entry for every query (tensor-core GEMM),
    top-k per query, attention per query over its selection and causal window."""
    import torch
    from long_context_hybrid_02_b300 import binding as B
    from long_context_hybrid_02_b300 import synth
    from long_context_hybrid_02_b300.pipeline import HybridLayer
    tok = synth.make_tokens(w, dev)
    qry = synth.make_queries(w, dev)
    layer = HybridLayer(w, tok, dev)
    layer.build_cache()
    # the chunk's tokens are positions L0 .. L-1: the blocks they complete are
    # compressed inside every step (rewriting the same entries each time)
    L0 = w.L - w.Tq
    blk0, n_blk_chunk = L0 // w.m, w.L // w.m - L0 // w.m
    blk_chunk = torch.full((w.B,), blk0, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    names = ["compress", "index", "topk", "attention"]
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(len(names) + 1)]
    ws = (layer.ws.data_ptr(), layer.ws.numel())

    def step(marks: bool):
        s = stream.cuda_stream
        ev[0].record(stream)
        layer.compress(blk_chunk, n_blk_chunk, s)
        if marks:
            ev[1].record(stream)
        B.csa_index_scores(layer.p, qry["qI"], qry["w_idx"], layer.cki, layer.n_cap, qry["q_pos"],
                           w.Tq, layer.scores, s)
        if marks:
            ev[2].record(stream)
        B.csa_topk(layer.p, layer.scores, layer.n_cap, qry["q_pos"], w.Tq, layer.idx, ws, s)
        if marks:
            ev[3].record(stream)
        B.hybrid_attn_prefill(layer.p, qry["q"], qry["q_pos"], w.Tq, layer.ck, layer.cv,
                              layer.n_cap, layer.idx, tok["k_tok"], tok["v_tok"], layer.tok_cap,
                              layer.o, layer.lse, ws, s)
        ev[4].record(stream)

    with torch.cuda.stream(stream):
        step(True)
    torch.cuda.synchronize()
    graphs = {}
    for marks in (False, True):
        g = torch.cuda.CUDAGraph()
        c0 = B.ha_launch_count()
        with torch.cuda.graph(g, stream=stream):
            step(marks)
        graphs[marks] = g
        launches_per_step = B.ha_launch_count() - c0
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def timed(g, k):
        tot, per = [], []
        for i in range(k):
            flush_w.fill_(i & 0xFF)
            torch.sum(flush_r, dim=0, out=flush_out)
            g.replay()
            torch.cuda.synchronize()
            tot.append(ev[0].elapsed_time(ev[len(names)]))
            if g is graphs[True]:
                per.append([ev[j].elapsed_time(ev[j + 1]) for j in range(len(names))])
        return tot, per

    for _ in range(args.warmup):
        graphs[False].replay()
        graphs[True].replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    with ClockSampler(dev) as clocks:
        t_wall0 = time.perf_counter()
        tot, _ = timed(graphs[False], args.steps)
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    tokens = w.B * w.Tq * world * args.steps
    value = tokens / (max_over_ranks(sum(tot), dev, dist, world) / 1e3)
    step_ms = sum(tot) / len(tot)
    tot_marked, per = timed(graphs[True], args.steps)
    kern_ms = {n: sum(p[j] for p in per) / len(per) for j, n in enumerate(names)}

    # algorithmic flops: attention 4*H*d per (query, key); indexer 2*H_I*d_I per (query, entry)
    pos = qry["q_pos"].to("cpu").long()
    t = pos.reshape(-1)
    ne = torch.clamp(t + 1 - w.n_win, min=0) // w.m
    keys = torch.clamp(ne, max=w.k) + torch.clamp(t + 1, max=w.n_win)
    attn_flops = float(4 * w.H * w.d * keys.sum().item())
    idx_flops = float(2 * w.H_I * w.d_I * ne.sum().item())
    pk = peaks()
    att_tf = attn_flops / (kern_ms["attention"] * 1e-3) / 1e12
    idx_tf = idx_flops / (kern_ms["index"] * 1e-3) / 1e12
    # one roofline entry per tensor-core kernel; `roofline` is the one with the larger
    # share of the step (the indexer on this workload)
    full_size = args.ctx == 0 and args.batch == 0
    entries = {}
    for name, tf, fl, src in (("index", idx_tf, idx_flops, "indexer_tc.cu"),
                              ("attention", att_tf, attn_flops, "attention_tc.cu")):
        entries[name] = {
            "bound": "tensor", "kernel": name, "achieved": round(tf, 1),
            "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(tf / pk["bf16_tflops"], 4),
            "traffic": profiled_traffic(args.workload if full_size else None, name, src),
            "algorithmic_flops": fl, "ms": round(kern_ms[name], 5),
            "peak_source": pk["source"] + " (MEASURED_PEAKS.json bf16_tflops, burst)"}
    dom = "index" if kern_ms["index"] >= kern_ms["attention"] else "attention"
    roofline = entries[dom]
    roofline_other = entries["attention" if dom == "index" else "index"]

    # end to end: the chunk's token rows and queries from pinned host memory, outputs back
    h_in = {k: host_buffer_like(qry[k], True) for k in ("q", "qI", "w_idx")}
    for k in h_in:
        h_in[k].copy_(qry[k])
    tok_names = ("k_tok", "v_tok", "ki_tok", "gate")
    for k in tok_names:
        h_in["chunk_" + k] = host_buffer_like(tok[k][:, L0:w.L], True)
        h_in["chunk_" + k].copy_(tok[k][:, L0:w.L])
    h_out = host_buffer_like(layer.o, False)
    h2d = sum(x.numel() * x.element_size() for x in h_in.values())
    d2h = h_out.numel() * h_out.element_size()
    qside = torch.cuda.Stream(device=dev)
    oside = torch.cuda.Stream(device=dev)
    n_sub = 8 if w.B == 1 and w.Tq % 8 == 0 else 1      # attention sub-chunks (B = 1: contiguous)
    sub = w.Tq // n_sub
    qfork = torch.cuda.Event()
    q_ready = [torch.cuda.Event() for _ in range(n_sub)]
    o_ready = [torch.cuda.Event() for _ in range(n_sub)]
    o_done = torch.cuda.Event()

    def e2e_step():
        """The chunk through the public API with its host copies, as one graph.  The
        chunk's token rows and the indexer's inputs are copied first; scoring and
        selection run over the whole chunk; the attention runs in sub-chunks of
        queries (the same call on a range of rows), each starting once its part of
        q has arrived (q is copied on a branch of its own right after the indexer's
        inputs) and each sending its part of o back on another branch while the
        next sub-chunk computes."""
        s = stream.cuda_stream
        for k in tok_names:
            tok[k][:, L0:w.L].copy_(h_in["chunk_" + k], non_blocking=True)
        for k in ("qI", "w_idx"):
            qry[k].copy_(h_in[k], non_blocking=True)
        # q follows the indexer's inputs on the link, so that scoring starts as soon
        # as they are in (together they would share the link's bandwidth)
        qfork.record(stream)
        qside.wait_event(qfork)
        with torch.cuda.stream(qside):
            for c in range(n_sub):
                qry["q"][:, c * sub:(c + 1) * sub].copy_(h_in["q"][:, c * sub:(c + 1) * sub],
                                                         non_blocking=True)
                q_ready[c].record(qside)
        layer.compress(blk_chunk, n_blk_chunk, s)
        B.csa_index_scores(layer.p, qry["qI"], qry["w_idx"], layer.cki, layer.n_cap, qry["q_pos"],
                           w.Tq, layer.scores, s)
        B.csa_topk(layer.p, layer.scores, layer.n_cap, qry["q_pos"], w.Tq, layer.idx, ws, s)
        for c in range(n_sub):
            r = slice(c * sub, (c + 1) * sub)
            stream.wait_event(q_ready[c])
            B.hybrid_attn_prefill(layer.p, qry["q"][:, r], qry["q_pos"][:, r], sub, layer.ck,
                                  layer.cv, layer.n_cap, layer.idx[:, r], tok["k_tok"],
                                  tok["v_tok"], layer.tok_cap, layer.o[:, r], layer.lse[:, r],
                                  ws, s)
            o_ready[c].record(stream)
            oside.wait_event(o_ready[c])
            with torch.cuda.stream(oside):
                h_out[:, r].copy_(layer.o[:, r], non_blocking=True)
        o_done.record(oside)
        stream.wait_event(o_done)

    with torch.cuda.stream(stream):
        e2e_step()                                  # eager warm-up
    torch.cuda.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        e2e_step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for i in range(args.steps):
        flush_w.fill_(i & 0xFF)
        torch.sum(flush_r, dim=0, out=flush_out)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            g_e2e.replay()
            e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_value = w.B * w.Tq * world * args.steps / (max_over_ranks(sum(e2e_ms), dev, dist, world) / 1e3)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok_h = {k: v[:1].to("cpu") for k, v in tok.items()}
        qry_h = {k: v[:1].to("cpu") for k, v in qry.items()}
        done, el, threads = oracle_prefill_sample(w, tok_h, qry_h, args.cpu_seconds)
        cpu = {"value": done / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "host_cpus": len(os.sched_getaffinity(0)),
               "sample": f"{done} prefill queries of sequence 0 (from the end of the chunk), "
                         f"{el:.1f}s; caches built untimed"}
    line = {
        "metric": "prefill tokens/s (one layer, one chunk)",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Gaussian drawn on the device)",
        "config": workload_config(w, L2_FLUSHED, GRAPH_TIMING),
        "clocks": clocks.summary(),
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "timing": "per step: pinned-host copies of the chunk's token rows (K, V, indexer "
                          "keys, gates) and queries, the step (compression of the blocks the "
                          "chunk completes first) and the copy of o back, one graph between "
                          "CUDA events; q copied after the indexer's inputs, beside "
                          "compression, scoring and selection, "
                          "attention in 8 sub-chunks of queries whose outputs are copied back "
                          "beside the next; L2 flushed before every step"},
        "gpu_launches": int(launches_per_step) * args.steps,
        "roofline": roofline,
        "roofline_" + roofline_other["kernel"]: roofline_other,
        "indexer_tflops": round(idx_tf, 1),
        "indexer_frac_of_sustained": (round(idx_tf / pk["bf16_tflops_sustained"], 4)
                                      if pk.get("bf16_tflops_sustained") else None),
        "cpu_baseline": cpu,
        "kernel_ms": {k: round(v, 5) for k, v in kern_ms.items()},
        "ms_per_step_with_kernel_events": round(sum(tot_marked) / len(tot_marked), 5),
        "wall_s_timed": round(t_wall, 3),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


# ----------------------------------------------------------------------------- GPU arm
def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        run_reference(args, rank)
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from long_context_hybrid_02_b300 import binding as B
    from long_context_hybrid_02_b300 import build as bld
    from long_context_hybrid_02_b300 import synth
    from long_context_hybrid_02_b300.pipeline import HybridLayer
    if not os.path.exists(bld.LIB):
        bld.build()
    B.load_library()
    w = scaled_workload(synth.WORKLOADS[args.workload], args)
    if not w.decode:
        return run_prefill(args, w, dev, world, rank, dist)
    tok = synth.make_tokens(w, dev)
    qry = synth.make_queries(w, dev)
    if w.plant_frac > 0:
        synth.plant_blocks(w, tok, qry, max(0, w.L - w.n_win) // w.m)
    layer = HybridLayer(w, tok, dev)
    layer.build_cache()
    bulk = bulk_compress_rate(w, layer, dev)
    recall = (fp4_indexer_recall(w, tok, qry, layer, dev)
              if w.kind == "csa" and w.fmt & 2 else None)
    new_blk = torch.full((w.B,), (w.L // w.m) - 1 if w.L % w.m == 0 else -1, dtype=torch.int32,
                         device=dev)
    q = qry["q"][:, 0].contiguous()
    stream = torch.cuda.Stream(device=dev)
    names = ["compress", "index", "topk", "attention"] if w.kind == "csa" else ["compress", "attention"]
    n_ev = len(names) + 1
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n_ev)]

    side = torch.cuda.Stream(device=dev)
    join = torch.cuda.Event()
    # Under the disjoint rule with n_win >= m the newest complete block lies inside
    # the query's window and is not eligible, so in the end-to-end step its
    # compression runs beside index / top-k / attention.
    concurrent_compress = layer.p.elig == B.ELIG_DISJOINT and w.n_win >= w.m

    def step(marks: bool):
        """One decode step.  The first and last events are always recorded.  Without
        marks (the headline) the step is one fused library call, csa_decode_step /
        hca_decode_step: compress the block the newest token completes, score,
        select, attend, chained on the stream.  With marks the same kernels run as
        the separate calls, one after the other, with an event between every two
        (the per-kernel breakdown: a recorded event between two kernels also keeps
        the second from starting early)."""
        s = stream.cuda_stream
        ev[0].record(stream)
        if not marks:
            layer.decode_step_fused(q, qry["ctx_len"], qry.get("qI"), qry.get("w_idx"), s)
            ev[n_ev - 1].record(stream)
            return
        layer.compress(new_blk, 1, s)
        ev[1].record(stream)
        if w.kind == "csa":
            B.csa_index_scores(layer.p, qry["qI"], qry["w_idx"], layer.cki, layer.n_cap,
                               qry["q_pos"], 1, layer.scores, s)
            ev[2].record(stream)
            B.csa_topk(layer.p, layer.scores, layer.n_cap, qry["q_pos"], 1, layer.idx,
                       (layer.ws.data_ptr(), layer.ws.numel()), s)
            ev[3].record(stream)
            idx = layer.idx
        else:
            idx = None
        B.hybrid_attn_decode(layer.p, q, layer.ck, layer.cv, layer.n_cap, idx, tok["k_tok"],
                             tok["v_tok"], layer.tok_cap, qry["ctx_len"], layer.o, layer.lse,
                             (layer.ws.data_ptr(), layer.ws.numel()), s)
        ev[n_ev - 1].record(stream)

    # eager warm-up (sets kernel attributes), then capture both graphs
    with torch.cuda.stream(stream):
        step(True)
        step(False)
    torch.cuda.synchronize()
    graphs = {}
    for marks in (False, True):
        g = torch.cuda.CUDAGraph()
        c0 = B.ha_launch_count()
        with torch.cuda.graph(g, stream=stream):
            step(marks)
        graphs[marks] = g
        launches_per_step = B.ha_launch_count() - c0
    graph = graphs[False]
    # L2 flush before every timed step: write 256 MiB, then read another 256 MiB, so
    # that neither our data nor dirty lines of the write are left in L2 (a write-
    # only flush leaves 126 MB of dirty lines whose write-back would share DRAM
    # with the timed step)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device=dev)
    flush_out = torch.empty((), dtype=torch.float32, device=dev)

    def flush(i):
        flush_w.fill_(i & 0xFF)
        torch.sum(flush_r, dim=0, out=flush_out)

    def timed(g, k):
        per = [[0.0] * (n_ev - 1) for _ in range(k)]
        tot = []
        for i in range(k):
            flush(i)
            g.replay()
            torch.cuda.synchronize()
            if g is graphs[True]:
                for j in range(n_ev - 1):
                    per[i][j] = ev[j].elapsed_time(ev[j + 1])
            tot.append(ev[0].elapsed_time(ev[n_ev - 1]))
        return tot, per

    for _ in range(args.warmup):
        flush(0)
        graph.replay()
        graphs[True].replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clocks:
        t_wall0 = time.perf_counter()
        tot, _ = timed(graph, args.steps)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = sum(tot) / len(tot)
    total_ms = max_over_ranks(sum(tot), dev, dist, world)
    tokens = w.B * world * args.steps
    value = tokens / (total_ms / 1e3)
    # per-kernel breakdown: the same steps with an event between every two calls
    tot_marked, per = timed(graphs[True], args.steps)
    kern_ms = {n: sum(p[j] for p in per) / len(per) for j, n in enumerate(names)}

    # ---- roofline of the dominant kernel (largest share of the step)
    ne = max(0, w.L - w.n_win) // w.m          # entries visible to the decode query
    nbytes = step_bytes(w, ne, min(w.n_win, w.L))
    dom = max(kern_ms, key=kern_ms.get)
    pk = peaks()
    achieved = nbytes[dom] / (kern_ms[dom] * 1e-3) / 1e9
    src_of = {"compress": "compress.cu", "index": "indexer_tc.cu", "topk": "topk.cu",
              "attention": "attention_tc.cu"}
    full_size = args.ctx == 0 and args.batch == 0
    traffic = profiled_traffic(args.workload if full_size else None, dom, src_of[dom])
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1),
                "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": traffic, "algorithmic_bytes": nbytes[dom],
                "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs)",
                # the same launch on the DRAM bytes ncu counted, and against the
                # part's nominal 7.7 TB/s
                "dram_gbs": (round(traffic / (kern_ms[dom] * 1e-3) / 1e9, 1)
                             if traffic is not None else None),
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4)}

    # ---- end to end through the public API: pinned host inputs -> step -> host output
    # The step's small inputs (the indexer's query and weights, the newest token's
    # rows) travel in one packed host-to-device copy; q (read only by the
    # attention) in a copy of its own beside scoring and selection.
    h_q = host_buffer_like(q, True)
    h_q.copy_(q)
    row = (w.L - 1) % layer.tok_cap
    small = {}
    if w.kind == "csa":
        small["qI"] = qry["qI"]
        small["w_idx"] = qry["w_idx"]
    for kname in (("k_tok", "v_tok", "ki_tok") if w.kind == "csa" else ("k_tok", "v_tok")):
        small["new_" + kname] = tok[kname][:, row]
    small["new_gate"] = tok["gate"][:, row]
    offs, total = {}, 0
    for kname, t in small.items():
        offs[kname] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    h_pack = B.host_empty((total,), torch.uint8, write_combined=True)
    d_pack = torch.empty(total, dtype=torch.uint8, device=dev)
    d_view = {}
    for kname, t in small.items():
        nb = t.numel() * t.element_size()
        d_view[kname] = d_pack[offs[kname]:offs[kname] + nb].view(t.dtype).reshape(t.shape)
        h_pack[offs[kname]:offs[kname] + nb].view(t.dtype).reshape(t.shape).copy_(t)
    h_out = host_buffer_like(layer.o, False)
    h2d = total + h_q.numel() * h_q.element_size()
    d2h = h_out.numel() * h_out.element_size()
    qside = torch.cuda.Stream(device=dev)
    qjoin, tok_ready = torch.cuda.Event(), torch.cuda.Event()
    pack_ready = torch.cuda.Event()
    tok_names = [kname for kname in small if kname.startswith("new_")]

    def e2e_step():
        """One decode step through the public API with its own host copies, as one
        graph: the packed small inputs are copied first on the main stream, then
        the newest token's rows are put into the per-token caches on a side branch
        ahead of the compression that reads them (the attention waits for them: the
        window holds the newest token); q is copied after the packed inputs on a
        branch of its own, beside scoring and selection; o is copied back at the
        end."""
        s = stream.cuda_stream
        d_pack.copy_(h_pack, non_blocking=True)
        pack_ready.record(stream)
        # q follows the packed inputs on the link (together they would share its
        # bandwidth and delay scoring)
        qside.wait_event(pack_ready)
        with torch.cuda.stream(qside):
            q.copy_(h_q, non_blocking=True)
        qjoin.record(qside)
        side.wait_event(pack_ready)
        with torch.cuda.stream(side):
            for kname in tok_names:
                tok[kname[4:]][:, row].copy_(d_view[kname], non_blocking=True)
        tok_ready.record(side)
        if concurrent_compress:
            layer.compress(new_blk, 1, side.cuda_stream)
            join.record(side)
        else:
            stream.wait_event(tok_ready)
            layer.compress(new_blk, 1, s)
        if w.kind == "csa":
            B.csa_index_scores(layer.p, d_view["qI"], d_view["w_idx"], layer.cki, layer.n_cap,
                               qry["q_pos"], 1, layer.scores, s)
            B.csa_topk(layer.p, layer.scores, layer.n_cap, qry["q_pos"], 1, layer.idx,
                       (layer.ws.data_ptr(), layer.ws.numel()), s)
        stream.wait_event(qjoin)
        stream.wait_event(tok_ready)
        B.hybrid_attn_decode(layer.p, q, layer.ck, layer.cv, layer.n_cap,
                             layer.idx if w.kind == "csa" else None, tok["k_tok"], tok["v_tok"],
                             layer.tok_cap, qry["ctx_len"], layer.o, layer.lse,
                             (layer.ws.data_ptr(), layer.ws.numel()), s)
        if concurrent_compress:
            stream.wait_event(join)
        h_out.copy_(layer.o, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()                                  # eager warm-up
    torch.cuda.synchronize()
    g_e2e = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_e2e, stream=stream):
        e2e_step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = []
    for i in range(args.steps):
        flush(i)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            e0.record(stream)
            g_e2e.replay()
            e1.record(stream)
        e1.synchronize()
        e2e_ms.append(e0.elapsed_time(e1))
    e2e_value = tokens / (max_over_ranks(sum(e2e_ms), dev, dist, world) / 1e3)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n_seq = 2
        tok_h = {k: v[:n_seq].to("cpu") for k, v in tok.items()}
        qry_h = {k: v[:n_seq].to("cpu") for k, v in qry.items()}
        done, el, threads, _ = oracle_sample(w, tok_h, qry_h, n_seq, args.cpu_seconds)
        cpu = {"value": done / el, "unit": "tokens/s", "cores": threads, "kind": "oracle",
               "host_cpus": len(os.sched_getaffinity(0)),
               "sample": f"{done} decode tokens: sequences 0..{n_seq - 1} of the same inputs "
                         f"(host copies) decoded repeatedly for {el:.1f}s; caches built untimed"}

    clk = clocks.summary()
    line = {
        "metric": "decode tokens/s (one layer, all sequences)",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32",
        "data": "synthetic (seeded Gaussian drawn on the device)",
        "config": workload_config(w, L2_FLUSHED, GRAPH_TIMING),
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "timing": "per step, one graph between CUDA events: the step's small inputs "
                          "(indexer query and weights, the newest token's rows) in one packed "
                          "copy from page-locked host memory, q in a copy of its own beside "
                          "scoring and selection, the separate library calls, the copy of o "
                          "back; L2 flushed before every step"},
        "gpu_launches": int(launches_per_step) * args.steps,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "kernel_ms": {k: round(v, 5) for k, v in kern_ms.items()},
        "bulk_compress": bulk,
        "indexer_recall": recall,
        "ms_per_step_with_kernel_events": round(sum(tot_marked) / len(tot_marked), 5),
        "step_algorithmic_gbs": round(sum(nbytes.values()) / (step_ms * 1e-3) / 1e9, 1),
        "wall_s_timed": round(t_wall, 3),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

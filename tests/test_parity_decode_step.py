"""The fused decode steps (csa_decode_step, hca_decode_step) and the cache state.

1. A fused step gives bit for bit what the separate calls give in the method's
   order (compress the block the newest token completes, score, select, attend):
   the same kernels, only chained differently.  Contexts that do and do not
   complete a block sit in one batch; the CUDA-core (float32) and tensor-core
   (bfloat16, 64 heads x 512, indexer 64 x 128) paths are both covered.
2. The state manager ("DeepSeek-V4 深度研究剖析" §11.4: compressed caches, indexer
   cache, window state and the tail tokens of unfinished blocks): ragged appends of
   new tokens into ring-buffered per-token caches, each compressing the blocks it
   completes, then fused decode steps, checked after every step against the
   oracle run on the whole token history.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B
from long_context_hybrid_02_b300 import synth
from long_context_hybrid_02_b300.cache_state import CacheState
from long_context_hybrid_02_b300.pipeline import HybridLayer
from tests._harness import (assert_close, assert_lse_close, assert_sorted_unique,
                            assert_topk_match, np64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _layer_pair(w, ctx):
    """Two layers over the same per-token caches with identical compressed caches
    (every complete block compressed, then each sequence's newest block wiped so
    that a step has to write it)."""
    tok = synth.make_tokens(w, DEV)
    a, b = HybridLayer(w, tok, DEV), HybridLayer(w, tok, DEV)
    for lay in (a, b):
        lay.build_cache()
        for s, c in enumerate(ctx):
            if c % w.m == 0 and c > 0:
                for t in ("ck", "cv", "cki"):
                    buf = getattr(lay, t)
                    if buf is not None:
                        buf[s, c // w.m - 1].fill_(7.0)
    return tok, a, b


def _queries(w, ctx):
    qry = synth.make_queries(w, DEV)
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    qry["ctx_len"] = ctx_t
    qry["q_pos"] = (ctx_t - 1).reshape(w.B, 1).contiguous()
    return qry


@pytest.mark.parametrize("name,ctx", [
    ("tiny_csa", [1024, 1023, 1020, 130, 129, 128, 4, 1]),
    ("csa_bf16", [16384, 16383, 16000, 12345, 8192, 4097, 300, 132]),
])
def test_csa_step_equals_the_separate_calls(name, ctx):
    if name == "tiny_csa":
        w = synth.WORKLOADS["tiny_csa"].scaled(B=len(ctx))
    else:
        w = synth.WORKLOADS["csa_decode_64k"].scaled(B=len(ctx), L=16384)
    tok, sep, fus = _layer_pair(w, ctx)
    qry = _queries(w, ctx)
    q = qry["q"][:, 0].contiguous()
    # separate calls: compress the newest block, then index, top-k, attention
    newest = torch.tensor([c // w.m - 1 if c % w.m == 0 else -1 for c in ctx], dtype=torch.int32,
                          device=DEV)
    sep.compress(newest, 1)
    ws = (sep.ws.data_ptr(), sep.ws.numel())
    B.csa_index_scores(sep.p, qry["qI"], qry["w_idx"], sep.cki, sep.n_cap, qry["q_pos"], 1, sep.scores)
    B.csa_topk(sep.p, sep.scores, sep.n_cap, qry["q_pos"], 1, sep.idx, ws)
    B.hybrid_attn_decode(sep.p, q, sep.ck, sep.cv, sep.n_cap, sep.idx, tok["k_tok"], tok["v_tok"],
                         sep.tok_cap, qry["ctx_len"], sep.o, sep.lse, ws)
    B.ha_device_error(clear=True)
    fus.decode_step_fused(q, qry["ctx_len"], qry["qI"], qry["w_idx"])
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    for t in ("ck", "cv", "cki"):
        assert torch.equal(getattr(sep, t), getattr(fus, t)), t
    for s, c in enumerate(ctx):
        ne = O.n_eligible(c - 1, w.n_win, w.m)
        assert torch.equal(sep.scores[s, 0, :ne], fus.scores[s, 0, :ne]), s
    assert torch.equal(sep.idx, fus.idx)
    assert torch.equal(sep.o, fus.o)
    assert torch.equal(sep.lse, fus.lse)


@pytest.mark.parametrize("name,ctx", [
    ("tiny_hca", [1024, 1023, 896, 200, 128, 1]),
    ("hca_bf16", [131072, 131071, 130944, 65536, 20000, 129]),
])
def test_hca_step_equals_the_separate_calls(name, ctx):
    if name == "tiny_hca":
        w = synth.WORKLOADS["tiny_hca"].scaled(B=len(ctx))
    else:
        w = synth.WORKLOADS["hca_decode_128k"].scaled(B=len(ctx))
    tok, sep, fus = _layer_pair(w, ctx)
    qry = _queries(w, ctx)
    q = qry["q"][:, 0].contiguous()
    newest = torch.tensor([c // w.m - 1 if c % w.m == 0 else -1 for c in ctx], dtype=torch.int32,
                          device=DEV)
    sep.compress(newest, 1)
    B.hybrid_attn_decode(sep.p, q, sep.ck, sep.cv, sep.n_cap, None, tok["k_tok"], tok["v_tok"],
                         sep.tok_cap, qry["ctx_len"], sep.o, sep.lse, (sep.ws.data_ptr(), sep.ws.numel()))
    B.ha_device_error(clear=True)
    fus.decode_step_fused(q, qry["ctx_len"])
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    assert torch.equal(sep.ck, fus.ck) and torch.equal(sep.cv, fus.cv)
    assert torch.equal(sep.o, fus.o)
    assert torch.equal(sep.lse, fus.lse)


def test_csa_step_matches_the_oracle_on_its_own_caches():
    """Two sequences of the 64K workload's shape (16K tokens), the oracle compressing
    every block itself and running compress -> index -> top-k -> attend in float64."""
    w = synth.WORKLOADS["csa_decode_64k"].scaled(B=2, L=16384)
    ctx = [16384, 16382]
    tok = synth.make_tokens(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache(n_blk=w.n_blocks - 1)        # the newest block is the step's to write
    qry = _queries(w, ctx)
    layer.decode_step_fused(qry["q"][:, 0].contiguous(), qry["ctx_len"], qry["qI"], qry["w_idx"])
    torch.cuda.synchronize()
    for b, c in enumerate(ctx):
        t = c - 1
        g = np64(tok["gate"][b, :c])
        K, V = np64(tok["k_tok"][b, :c]), np64(tok["v_tok"][b, :c])
        nb = c // w.m
        ck, cv = O.compress(K, g, w.m, 0, nb, "bf16"), O.compress(V, g, w.m, 0, nb, "bf16")
        cki = O.compress(np64(tok["ki_tok"][b, :c]), g, w.m, 0, nb, "bf16")
        assert_close(np64(layer.ck[b, :nb]), ck, "bf16", f"ck[{b}]")
        assert_close(np64(layer.cki[b, :nb]), cki, "bf16", f"cki[{b}]")
        ne = O.n_eligible(t, w.n_win, w.m)
        ref_scores = O.index_scores(np64(qry["qI"][b, 0]), np64(qry["w_idx"][b, 0]),
                                    np64(layer.cki[b, :ne]))
        gi = layer.idx[b, 0].cpu().numpy()
        assert_sorted_unique(gi, ne, w.k, f"idx[{b}]")
        assert_topk_match(gi, O.topk_select(ref_scores, w.k), ref_scores, w.k, f"top-k[{b}]")
        ro, rl = O.prefill_query(np64(qry["q"][b, 0]), gi, ck, cv, K, V, t, n_win=w.n_win, m=w.m,
                                 scale=1 / math.sqrt(w.d))
        assert_close(np64(layer.o[b, 0]), ro, "bf16", f"o[{b}]")
        assert_lse_close(np64(layer.lse[b, 0]), rl, "bf16", f"lse[{b}]")


# ------------------------------------------------------------------ the cache state
def _history(w, L_max, seed):
    """Every token row a sequence will ever receive, drawn up front (device)."""
    wl = w.scaled(L=L_max, seed=seed)
    return synth.make_tokens(wl, DEV)


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_ragged_appends_into_ring_caches_then_decode_steps(kind):
    """Three sequences, per-token caches in a ring of 512 slots: ragged prefill
    appends (each compressing the blocks it completes, -1 for sequences that
    complete none), then decode steps through the fused call; after each step
    every sequence is checked against the oracle run on its whole token history."""
    m = 4 if kind == "csa" else 128
    base = synth.WORKLOADS["csa_decode_64k" if kind == "csa" else "hca_decode_128k"]
    w = base.scaled(B=3, L=512, k=64, rope_dims=0)
    tok_cap, L_max = 512, 2048
    n_cap = L_max // m
    hist = _history(w, L_max, seed=21)
    ring = {name: torch.zeros((w.B, tok_cap) + t.shape[2:], dtype=t.dtype, device=DEV)
            for name, t in hist.items()}
    state = CacheState(w.B, m, w.n_win, tok_cap, n_cap)
    layer = HybridLayer(w, ring, DEV, n_cap=n_cap, tok_cap=tok_cap, state=state)
    for buf in (layer.ck, layer.cv, layer.cki):
        if buf is not None:
            buf.fill_(float("nan"))                 # entries never written must never be read
    chunks = [[300, 128, 5], [200, 385, 381], [57, 0, 100], [385, 200, 129]]
    ctx = np.zeros(w.B, dtype=np.int64)
    for n_new in chunks:
        rows = {}
        for name, t in hist.items():
            part = torch.zeros((w.B, max(n_new)) + t.shape[2:], dtype=t.dtype, device=DEV)
            for b in range(w.B):
                part[b, :n_new[b]] = t[b, ctx[b]:ctx[b] + n_new[b]]
            rows[name] = part
        ctx = layer.append(rows, n_new)
    qry = synth.make_queries(w.scaled(seed=22), DEV)
    scale = 1 / math.sqrt(w.d)
    for step in range(6):
        rows = {name: torch.stack([t[b, ctx[b]:ctx[b] + 1] for b in range(w.B)])
                for name, t in hist.items()}
        # the step compresses the block its newest token completes itself; the host
        # state only advances (and still checks the ring)
        n_new = [1] * w.B
        slots = [state.slots(b, 1) for b in range(w.B)]
        state.append(n_new)
        for name, dst in ring.items():
            for b in range(w.B):
                dst[b, int(slots[b][0])] = rows[name][b, 0].to(dst.dtype)
        ctx = state.ctx.copy()
        ctx_len = torch.tensor(ctx, dtype=torch.int32, device=DEV)
        q = synth.gaussian((w.B, w.H, w.d), DEV, 300 + step, scale, w.torch_dtype)
        qI = w_idx = None
        if kind == "csa":
            qI = synth.gaussian((w.B, 1, w.H_I, w.d_I), DEV, 400 + step, 1 / math.sqrt(w.d_I),
                                w.torch_dtype)
            w_idx = qry["w_idx"]
        B.ha_device_error(clear=True)
        layer.decode_step_fused(q, ctx_len, qI, w_idx)
        torch.cuda.synchronize()
        assert B.ha_device_error() == 0
        for b in range(w.B):
            c = int(ctx[b])
            t = c - 1
            g = np64(hist["gate"][b, :c])
            K, V = np64(hist["k_tok"][b, :c]), np64(hist["v_tok"][b, :c])
            ne = O.n_eligible(t, w.n_win, m)
            ck = O.compress(K, g, m, 0, ne, "bf16")
            cv = O.compress(V, g, m, 0, ne, "bf16")
            assert_close(np64(layer.ck[b, :ne]), ck, "bf16", f"step {step} ck[{b}]")
            assert_close(np64(layer.cv[b, :ne]), cv, "bf16", f"step {step} cv[{b}]")
            if kind == "csa":
                cki = O.compress(np64(hist["ki_tok"][b, :c]), g, m, 0, ne, "bf16")
                assert_close(np64(layer.cki[b, :ne]), cki, "bf16", f"step {step} cki[{b}]")
                ref_scores = O.index_scores(np64(qI[b, 0]), np64(w_idx[b, 0]),
                                            np64(layer.cki[b, :ne]))
                gi = layer.idx[b, 0].cpu().numpy()
                assert_sorted_unique(gi, ne, w.k, f"step {step} idx[{b}]")
                assert_topk_match(gi, O.topk_select(ref_scores, w.k), ref_scores, w.k,
                                  f"step {step} top-k[{b}]")
                ro, rl = O.prefill_query(np64(q[b]), gi, ck, cv, K, V, t, n_win=w.n_win, m=m,
                                         scale=scale)
            else:
                ro, rl = O.prefill_query(np64(q[b]), None, ck, cv, K, V, t, n_win=w.n_win, m=m,
                                         scale=scale)
            assert_close(np64(layer.o[b, 0]), ro, "bf16", f"step {step} o[{b}]")
            assert_lse_close(np64(layer.lse[b, 0]), rl, "bf16", f"step {step} lse[{b}]")

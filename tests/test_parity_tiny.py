"""GPU vs oracle on the tiny float32 layers (whole workload, every output).

1 sequence of 1024 tokens, 8 query heads of dim 64, one shared K/V head, window
128, CSA m = 4 (256 entries, top-16) and HCA m' = 128 (8 entries), indexer 2 x 32.
Plus batched variants with per-sequence lengths that hit the edge cases
(context shorter than the window, exactly at block boundaries, empty context).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B
from long_context_hybrid_02_b300 import synth
from long_context_hybrid_02_b300.pipeline import HybridLayer, params_for
from tests._harness import (assert_close, assert_lse_close, assert_sorted_unique,
                            assert_topk_match, np64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def to_dev(d):
    return {k: v.to(DEV) for k, v in d.items()}


def oracle_caches(w, tok):
    """Oracle compression of every complete block of every sequence (storage-rounded)."""
    out = {"ck": [], "cv": [], "cki": []}
    for b in range(w.B):
        g = np64(tok["gate"][b])
        out["ck"].append(O.compress(np64(tok["k_tok"][b]), g, w.m, 0, w.n_blocks, w.dtype))
        out["cv"].append(O.compress(np64(tok["v_tok"][b]), g, w.m, 0, w.n_blocks, w.dtype))
        if w.kind == "csa":
            out["cki"].append(O.compress(np64(tok["ki_tok"][b]), g, w.m, 0, w.n_blocks, w.dtype))
    return out


@pytest.mark.parametrize("name", ["tiny_csa", "tiny_hca"])
def test_tiny_decode_step_end_to_end(name):
    w = synth.WORKLOADS[name]
    tok, qry = synth.make_tokens(w, "cpu"), synth.make_queries(w, "cpu")
    layer = HybridLayer(w, to_dev(tok), DEV)
    layer.build_cache()
    qd = to_dev(qry)
    new_blk = torch.full((w.B,), w.n_blocks - 1, dtype=torch.int32, device=DEV)
    layer.decode_step(qd["q"][:, 0], qd["ctx_len"], new_blk, qd.get("qI"), qd.get("w_idx"),
                      qd["q_pos"])
    torch.cuda.synchronize()
    ref = oracle_caches(w, tok)
    assert_close(np64(layer.ck[0]), ref["ck"][0], w.dtype, "ck")
    assert_close(np64(layer.cv[0]), ref["cv"][0], w.dtype, "cv")
    t = w.L - 1
    q = np64(qry["q"][0, 0])
    scale = 1 / math.sqrt(w.d)
    if w.kind == "csa":
        assert_close(np64(layer.cki[0]), ref["cki"][0], w.dtype, "cki")
        o, lse, idx, scores = O.csa_decode(q, np64(qry["qI"][0, 0]), np64(qry["w_idx"][0, 0]),
                                           ref["ck"][0], ref["cv"][0], ref["cki"][0],
                                           np64(tok["k_tok"][0]), np64(tok["v_tok"][0]), t,
                                           n_win=w.n_win, m=w.m, k=w.k, scale=scale)
        ne = O.n_eligible(t, w.n_win, w.m)
        assert_close(np64(layer.scores[0, 0, :ne]), scores, w.dtype, "scores")
        gi = layer.idx[0, 0].cpu().numpy()
        assert_sorted_unique(gi, ne, w.k, "idx")
        assert_topk_match(gi, idx, scores, w.k, "top-k")
    else:
        o, lse = O.hca_decode(q, ref["ck"][0], ref["cv"][0], np64(tok["k_tok"][0]),
                              np64(tok["v_tok"][0]), t, n_win=w.n_win, m=w.m, scale=scale)
    assert_close(np64(layer.o[0, 0]), o, w.dtype, "o")
    assert_lse_close(np64(layer.lse[0, 0]), lse, w.dtype, "lse")


def test_tiny_topk_stage_is_exact_on_identical_scores():
    """csa_topk on oracle-made float32 scores picks exactly the oracle's entries,
    including ties and NaN, for rows of several lengths."""
    w = synth.WORKLOADS["tiny_csa"].scaled(B=6)
    p = params_for(w)
    n_cap = 300
    rng = np.random.default_rng(0)
    s = np.round(rng.standard_normal((w.B, 1, n_cap)), 2).astype(np.float32)   # many ties
    s[2, 0, 5:40] = np.nan
    s[3, 0, :] = 1.0                                                             # all tied
    ctx = [1, 129, 200, 1024, 1024, 1300]
    q_pos = torch.tensor([[c - 1] for c in ctx], dtype=torch.int32, device=DEV)
    scores = torch.from_numpy(s).to(DEV)
    idx = torch.full((w.B, 1, w.k), -7, dtype=torch.int32, device=DEV)
    B.csa_topk(p, scores, n_cap, q_pos, 1, idx)
    torch.cuda.synchronize()
    for b, c in enumerate(ctx):
        ne = min(O.n_eligible(c - 1, w.n_win, w.m), n_cap)
        ref = O.topk_select(s[b, 0, :ne].astype(np.float64), w.k)
        assert idx[b, 0].cpu().numpy().tolist() == ref.tolist(), b


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_tiny_batched_edge_lengths(kind):
    """Per-sequence context lengths: empty, shorter than the window, at block and
    window boundaries, full.  Decode attention against the oracle for each."""
    base = synth.WORKLOADS["tiny_" + kind]
    w = base.scaled(B=7)
    ctx = [0, 1, 100, 128, 129, 128 + base.m, 1024]
    tok, qry = synth.make_tokens(w, "cpu"), synth.make_queries(w, "cpu")
    qry["ctx_len"] = torch.tensor(ctx, dtype=torch.int32)
    qry["q_pos"] = (qry["ctx_len"] - 1).reshape(-1, 1).to(torch.int32)
    layer = HybridLayer(w, to_dev(tok), DEV)
    layer.build_cache()
    qd = to_dev(qry)
    if kind == "csa":
        B.csa_index_scores(layer.p, qd["qI"], qd["w_idx"], layer.cki, layer.n_cap, qd["q_pos"], 1,
                           layer.scores)
        B.csa_topk(layer.p, layer.scores, layer.n_cap, qd["q_pos"], 1, layer.idx,
                   (layer.ws.data_ptr(), layer.ws.numel()))
    B.hybrid_attn_decode(layer.p, qd["q"][:, 0], layer.ck, layer.cv, layer.n_cap,
                         layer.idx if kind == "csa" else None, layer.tok["k_tok"],
                         layer.tok["v_tok"], layer.tok_cap, qd["ctx_len"], layer.o, layer.lse,
                         (layer.ws.data_ptr(), layer.ws.numel()))
    torch.cuda.synchronize()
    ref = oracle_caches(w, tok)
    scale = 1 / math.sqrt(w.d)
    for b, c in enumerate(ctx):
        q = np64(qry["q"][b, 0])
        if c == 0:
            assert (np64(layer.o[b, 0]) == 0).all()
            assert np.isneginf(np64(layer.lse[b, 0])).all()
            continue
        t = c - 1
        K, V = np64(tok["k_tok"][b]), np64(tok["v_tok"][b])
        if kind == "csa":
            o, lse, idx, scores = O.csa_decode(q, np64(qry["qI"][b, 0]), np64(qry["w_idx"][b, 0]),
                                               ref["ck"][b], ref["cv"][b], ref["cki"][b], K, V, t,
                                               n_win=w.n_win, m=w.m, k=w.k, scale=scale)
            assert_topk_match(layer.idx[b, 0].cpu().numpy(), idx, scores, w.k, f"top-k {b}")
        else:
            o, lse = O.hca_decode(q, ref["ck"][b], ref["cv"][b], K, V, t, n_win=w.n_win, m=w.m,
                                  scale=scale)
        assert_close(np64(layer.o[b, 0]), o, w.dtype, f"o[{b}]")
        assert_lse_close(np64(layer.lse[b, 0]), lse, w.dtype, f"lse[{b}]")


def test_tiny_decode_attention_stage_with_given_index_sets():
    """hybrid_attn_decode alone on generator-made index sets (unsorted, with -1 and
    out-of-range entries, which are ignored)."""
    w = synth.WORKLOADS["tiny_csa"].scaled(B=3)
    tok, qry = synth.make_tokens(w, "cpu"), synth.make_queries(w, "cpu")
    p = params_for(w)
    n_cap = w.n_blocks
    ck = synth.gaussian((w.B, n_cap, w.d), "cpu", 11, 1 / math.sqrt(w.d))
    cv = synth.gaussian((w.B, n_cap, w.d), "cpu", 12, 1 / math.sqrt(w.d))
    ne = O.n_eligible(w.L - 1, w.n_win, w.m)
    idx = synth.random_index_sets(w.B, 1, w.k, torch.full((w.B, 1), ne), "cpu", 5, pad_frac=0.25)
    idx = idx[:, 0].clone()
    idx[1] = idx[1].flip(0)                    # any order is accepted
    idx[2, 3] = ne + 5                         # ineligible: ignored
    idx[2, 4] = 10 ** 6                        # beyond n_cap: ignored
    o = torch.empty((w.B, w.H, w.d), dtype=torch.float32, device=DEV)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device=DEV)
    nb = B.ha_workspace_size(p, B.OP_DECODE, 1, n_cap, True)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    B.hybrid_attn_decode(p, qry["q"][:, 0].to(DEV), ck.to(DEV), cv.to(DEV), n_cap, idx.to(DEV),
                         tok["k_tok"].to(DEV), tok["v_tok"].to(DEV), w.L, qry["ctx_len"].to(DEV),
                         o, lse, ws)
    torch.cuda.synchronize()
    for b in range(w.B):
        # the raw set: the oracle itself ignores the -1 and ineligible entries
        ro, rl = O.prefill_query(np64(qry["q"][b, 0]), idx[b].numpy(), np64(ck[b]), np64(cv[b]),
                                 np64(tok["k_tok"][b]), np64(tok["v_tok"][b]), w.L - 1,
                                 n_win=w.n_win, m=w.m, scale=1 / math.sqrt(w.d))
        assert_close(np64(o[b]), ro, "f32", f"o[{b}]")
        assert_lse_close(np64(lse[b]), rl, "f32", f"lse[{b}]")


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_tiny_prefill_chunk(kind):
    """64 prefill queries at the end of the 1024-token context, each with its own
    selection and causal window (positions not block-aligned)."""
    w = synth.WORKLOADS["tiny_" + kind].scaled(Tq=64)
    tok, qry = synth.make_tokens(w, "cpu"), synth.make_queries(w, "cpu")
    layer = HybridLayer(w, to_dev(tok), DEV)
    layer.build_cache()
    qd = to_dev(qry)
    layer.prefill_chunk(qd["q"], qd["q_pos"], qd.get("qI"), qd.get("w_idx"))
    torch.cuda.synchronize()
    ref = oracle_caches(w, tok)
    K, V = np64(tok["k_tok"][0]), np64(tok["v_tok"][0])
    for i in range(w.Tq):
        t = int(qry["q_pos"][0, i])
        q = np64(qry["q"][0, i])
        if kind == "csa":
            o, lse, idx, scores = O.csa_decode(q, np64(qry["qI"][0, i]), np64(qry["w_idx"][0, i]),
                                               ref["ck"][0], ref["cv"][0], ref["cki"][0], K, V, t,
                                               n_win=w.n_win, m=w.m, k=w.k, scale=w.d ** -0.5)
            ne = O.n_eligible(t, w.n_win, w.m)
            assert_close(np64(layer.scores[0, i, :ne]), scores, w.dtype, f"scores[{i}]")
            assert_topk_match(layer.idx[0, i].cpu().numpy(), idx, scores, w.k, f"top-k[{i}]")
            gi = layer.idx[0, i].cpu().numpy()
            o, lse = O.prefill_query(q, gi, ref["ck"][0], ref["cv"][0], K, V, t, n_win=w.n_win,
                                     m=w.m, scale=w.d ** -0.5)
        else:
            o, lse = O.prefill_query(q, None, ref["ck"][0], ref["cv"][0], K, V, t, n_win=w.n_win,
                                     m=w.m, scale=w.d ** -0.5)
        assert_close(np64(layer.o[0, i]), o, w.dtype, f"o[{i}]")
        assert_lse_close(np64(layer.lse[0, i]), lse, w.dtype, f"lse[{i}]")


def test_decode_is_bitwise_repeatable_and_batch_invariant():
    """Deterministic kernels: the same sequence gives the same bits alone and inside
    a batch, and on a second run."""
    w = synth.WORKLOADS["tiny_csa"].scaled(B=4)
    tok, qry = synth.make_tokens(w, "cpu"), synth.make_queries(w, "cpu")
    layer = HybridLayer(w, to_dev(tok), DEV)
    layer.build_cache()
    qd = to_dev(qry)
    layer.decode_step(qd["q"][:, 0], qd["ctx_len"], None, qd["qI"], qd["w_idx"], qd["q_pos"])
    first = layer.o.clone()
    layer.decode_step(qd["q"][:, 0], qd["ctx_len"], None, qd["qI"], qd["w_idx"], qd["q_pos"])
    assert torch.equal(first, layer.o)
    w1 = w.scaled(B=1)
    one = HybridLayer(w1, {k: v[2:3].contiguous() for k, v in to_dev(tok).items()}, DEV)
    one.build_cache()
    one.decode_step(qd["q"][2:3, 0], qd["ctx_len"][2:3], None, qd["qI"][2:3], qd["w_idx"][2:3],
                    qd["q_pos"][2:3])
    torch.cuda.synchronize()
    assert torch.equal(one.idx[0], layer.idx[2])
    # the launch plan never depends on the batch, so the bits match across batches
    assert torch.equal(one.o[0], first[2])
    assert torch.equal(one.lse[0], layer.lse[2])

"""GPU vs oracle at the full prefill and million-token workloads, in the benchmark's
launch configuration.

CSA prefill: 4,096 new queries after a 131,072-token context (33,792 compressed
entries, top-512 per query, 64 heads x 512, indexer 64 x 128, bfloat16).
CSA decode 1M: 4 sequences x 1,048,576 tokens (262,144 entries scored per query,
top-1024, 128 heads), 1 % of the blocks planted with a query-aligned component.
HCA decode 1M: 4 sequences x 1,048,576 tokens (8,192 entries, all attended).

Every stage is checked on the very bytes its call consumed, each computed by the
oracle: sampled blocks of the compressor; full score rows and index sets of the
sampled queries (sets equal up to the 1e-6 band around the k-th oracle score);
attention over the index set the call used, plus the window.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import synth
from long_context_hybrid_02_b300.pipeline import HybridLayer
from tests._harness import (assert_close, assert_lse_close, assert_sorted_unique,
                            assert_topk_match, np64)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _check_blocks(w, tok, layer, b, blocks, names):
    for j in blocks:
        rows = slice(j * w.m, (j + 1) * w.m)
        g = np64(tok["gate"][b, rows])
        for name, cname in names:
            ref = O.compress(np64(tok[name][b, rows]), g, w.m, 0, 1, "bf16")[0]
            assert_close(np64(getattr(layer, cname)[b, j]), ref, "bf16", f"{cname}[{b},{j}]")


def _f32(t):
    """A bfloat16 device tensor as a float32 host array (exact)."""
    return t.float().cpu().numpy()


def _check_attention(w, q, idx, ck, cv, k_tok, v_tok, t, o, lse, what):
    """o/lse of one query against the oracle: the query's raw index set as the
    call consumed it (None: HCA, every eligible entry) + its window; the oracle
    ignores padding and ineligible entries itself.  Only the window's per-token
    rows are copied to the host."""
    lo = max(0, t - w.n_win + 1)
    idx = None if idx is None else idx.cpu().numpy()
    ro, rl = O.prefill_query(np64(q), idx, _f32(ck), _f32(cv), _f32(k_tok[lo:t + 1]),
                             _f32(v_tok[lo:t + 1]), t, n_win=w.n_win, m=w.m,
                             scale=1 / math.sqrt(q.shape[-1]), tok_base=lo)
    assert_close(np64(o), ro, "bf16", what + " o")
    assert_lse_close(np64(lse), rl, "bf16", what + " lse")


# ------------------------------------------------------------------ CSA prefill chunk
@pytest.fixture(scope="module")
def prefill():
    w = synth.WORKLOADS["csa_prefill_4k"]
    tok = synth.make_tokens(w, DEV)
    qry = synth.make_queries(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache()
    layer.prefill_chunk(qry["q"], qry["q_pos"], qry["qI"], qry["w_idx"])
    torch.cuda.synchronize()
    yield w, tok, qry, layer
    del layer, tok, qry
    torch.cuda.empty_cache()


SAMPLE_Q = (0, 1, 1000, 2047, 3333, 4095)


def test_prefill_compress_sampled_blocks(prefill):
    w, tok, qry, layer = prefill
    rng = np.random.default_rng(11)
    blocks = list(rng.integers(0, w.n_blocks, 24)) + [0, w.n_blocks - 1]
    _check_blocks(w, tok, layer, 0, blocks, (("k_tok", "ck"), ("v_tok", "cv"), ("ki_tok", "cki")))


def test_prefill_scores_and_topk_sampled_queries(prefill):
    w, tok, qry, layer = prefill
    cki = np64(layer.cki[0])
    for i in SAMPLE_Q:
        t = int(qry["q_pos"][0, i])
        ne = O.n_eligible(t, w.n_win, w.m)
        ref = O.index_scores(np64(qry["qI"][0, i]), np64(qry["w_idx"][0, i]), cki[:ne])
        got = np64(layer.scores[0, i, :ne])
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max())
        gi = layer.idx[0, i].cpu().numpy()
        assert_sorted_unique(gi, ne, w.k, f"idx[{i}]")
        assert_topk_match(gi, O.topk_select(ref, w.k), ref, w.k, f"top-k[{i}]")


def test_prefill_attention_sampled_queries(prefill):
    w, tok, qry, layer = prefill
    for i in SAMPLE_Q:
        t = int(qry["q_pos"][0, i])
        _check_attention(w, qry["q"][0, i], layer.idx[0, i], layer.ck[0], layer.cv[0],
                         tok["k_tok"][0], tok["v_tok"][0], t, layer.o[0, i], layer.lse[0, i],
                         f"[{i}]")


# ------------------------------------------------------------------ CSA decode, 1M tokens
@pytest.fixture(scope="module")
def csa_1m():
    w = synth.WORKLOADS["csa_decode_1m"]
    tok = synth.make_tokens(w, DEV)
    qry = synth.make_queries(w, DEV)
    ne = O.n_eligible(w.L - 1, w.n_win, w.m)
    planted = synth.plant_blocks(w, tok, qry, ne)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache()
    new_blk = torch.full((w.B,), w.n_blocks - 1, dtype=torch.int32, device=DEV)
    layer.decode_step(qry["q"][:, 0].contiguous(), qry["ctx_len"], new_blk, qry["qI"],
                      qry["w_idx"], qry["q_pos"])
    torch.cuda.synchronize()
    yield w, tok, qry, layer, planted
    del layer, tok, qry
    torch.cuda.empty_cache()


def test_1m_csa_compress_sampled_blocks(csa_1m):
    w, tok, qry, layer, planted = csa_1m
    rng = np.random.default_rng(12)
    for b in (0, 3):
        blocks = list(rng.integers(0, w.n_blocks, 12)) + [int(planted[b, 0]), w.n_blocks - 1]
        _check_blocks(w, tok, layer, b, blocks,
                      (("k_tok", "ck"), ("v_tok", "cv"), ("ki_tok", "cki")))


def test_1m_csa_scores_topk_and_planted_recall(csa_1m):
    """Full 262,143-entry score rows and top-1024 sets of every sequence; the planted
    blocks (+3 sigma on the query's direction) are what the selection picks."""
    w, tok, qry, layer, planted = csa_1m
    t = w.L - 1
    ne = O.n_eligible(t, w.n_win, w.m)
    for b in range(w.B):
        ref = O.index_scores(np64(qry["qI"][b, 0]), np64(qry["w_idx"][b, 0]), np64(layer.cki[b, :ne]))
        got = np64(layer.scores[b, 0, :ne])
        np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6 * np.abs(ref).max())
        gi = layer.idx[b, 0].cpu().numpy()
        assert_sorted_unique(gi, ne, w.k, f"idx[{b}]")
        assert_topk_match(gi, O.topk_select(ref, w.k), ref, w.k, f"top-k[{b}]")
        # diagnostic of the workload itself: most of the selection is planted blocks
        share = len(set(gi.tolist()) & set(planted[b].tolist())) / w.k
        print(f"sequence {b}: planted share of the top-{w.k} = {share:.3f}")
        assert share > 0.5, f"sequence {b}: only {share:.3f} of the selection is planted"


def test_1m_csa_attention(csa_1m):
    w, tok, qry, layer, planted = csa_1m
    t = w.L - 1
    for b in range(w.B):
        _check_attention(w, qry["q"][b, 0], layer.idx[b, 0], layer.ck[b], layer.cv[b],
                         tok["k_tok"][b], tok["v_tok"][b], t, layer.o[b, 0], layer.lse[b, 0],
                         f"[{b}]")


# ------------------------------------------------------------------ HCA decode, 1M tokens
@pytest.fixture(scope="module")
def hca_1m():
    w = synth.WORKLOADS["hca_decode_1m"]
    tok = synth.make_tokens(w, DEV)
    qry = synth.make_queries(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache()
    new_blk = torch.full((w.B,), w.n_blocks - 1, dtype=torch.int32, device=DEV)
    layer.decode_step(qry["q"][:, 0].contiguous(), qry["ctx_len"], new_blk, q_pos=qry["q_pos"])
    torch.cuda.synchronize()
    yield w, tok, qry, layer
    del layer, tok, qry
    torch.cuda.empty_cache()


def test_1m_hca_compress_and_attention(hca_1m):
    w, tok, qry, layer = hca_1m
    rng = np.random.default_rng(13)
    _check_blocks(w, tok, layer, 1, list(rng.integers(0, w.n_blocks, 6)) + [w.n_blocks - 1],
                  (("k_tok", "ck"), ("v_tok", "cv")))
    t = w.L - 1
    for b in range(w.B):
        _check_attention(w, qry["q"][b, 0], None, layer.ck[b], layer.cv[b], tok["k_tok"][b],
                         tok["v_tok"][b], t, layer.o[b, 0], layer.lse[b, 0], f"[{b}]")

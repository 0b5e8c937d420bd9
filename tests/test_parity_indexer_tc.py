"""Tensor-core indexer (bfloat16, 64 heads x 128 dims) against the oracle.

Shapes span several 128-entry tiles with ragged tails, sequences of different
lengths, decode (one query per sequence) and prefill query groups of 4 with a
partial last group, so that every branch of the tile walk is exercised.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B
from long_context_hybrid_02_b300 import synth
from tests._harness import assert_topk_match, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(B_, Tq, n_cap, positions, seed, k=64):
    p = B.make_params(B_, 1, 512, 128, 4, k, 64, 128, B.BF16)
    qI = synth.gaussian((B_, Tq, 64, 128), DEV, seed, 1 / math.sqrt(128), torch.bfloat16)
    w = torch.rand((B_, Tq, 64), generator=torch.Generator(DEV).manual_seed(seed), device=DEV)
    cki = synth.gaussian((B_, n_cap, 128), DEV, seed + 1, 1 / math.sqrt(128), torch.bfloat16)
    q_pos = torch.tensor(positions, dtype=torch.int32, device=DEV).reshape(B_, Tq)
    scores = torch.full((B_, Tq, n_cap), float("nan"), device=DEV)
    B.ha_device_error(clear=True)
    B.csa_index_scores(p, qI, w, cki, n_cap, q_pos, Tq, scores)
    idx = torch.empty((B_, Tq, k), dtype=torch.int32, device=DEV)
    B.csa_topk(p, scores, n_cap, q_pos, Tq, idx)
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    return qI, w, cki, q_pos, scores, idx


def _check(qI, w, cki, q_pos, scores, idx, k=64):
    B_, Tq, n_cap = scores.shape
    for b in range(B_):
        for t in range(Tq):
            pos = int(q_pos[b, t])
            ne = min(O.n_eligible(pos, 128, 4), n_cap)
            ref = O.index_scores(np64(qI[b, t]), np64(w[b, t]), np64(cki[b, :ne]))
            got = np64(scores[b, t, :ne])
            np.testing.assert_allclose(got, ref, rtol=1e-5, atol=1e-6 * max(1e-30, np.abs(ref).max(initial=0)))
            # nothing beyond the eligible prefix is written
            assert np.isnan(np64(scores[b, t, ne:])).all()
            assert_topk_match(idx[b, t].cpu().numpy(), O.topk_select(ref, k), ref, k, f"[{b},{t}]")


def test_tc_indexer_decode_ragged_sequences():
    # eligible entries per sequence: 0, 1, 127, 128, 129, 1000 (n_cap 1000, 8 tiles)
    pos = [100, 128 + 4 - 1, 128 + 4 * 127 - 1, 128 + 4 * 128 - 1, 128 + 4 * 129 - 1, 100000]
    r = _run(len(pos), 1, 1000, pos, seed=5)
    _check(*r)


def test_tc_indexer_prefill_groups_with_partial_tail():
    # 2 sequences x 10 queries (groups of 4, 4, 2), causal positions spanning tile edges
    L0 = 128 + 4 * 300
    pos = [[L0 + 37 * i for i in range(10)], [L0 + 500 + i for i in range(10)]]
    r = _run(2, 10, 900, [x for row in pos for x in row], seed=9)
    _check(*r)


def test_tc_indexer_many_sequences_uneven_split():
    # more tiles than CTAs with uneven per-CTA ranges crossing sequence boundaries
    rng = np.random.default_rng(3)
    pos = [int(x) for x in rng.integers(128, 128 + 4 * 3000, 40)]
    r = _run(40, 1, 3000, pos, seed=13)
    _check(*r)

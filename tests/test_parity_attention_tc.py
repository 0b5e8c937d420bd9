"""Tensor-core attention (bfloat16, head dim 512, 64-head groups) against the oracle.

The decode and prefill calls take this path whenever the storage is bfloat16,
d = 512 and H is a multiple of 64.  The cases cover what the key-list layout and
the split plan make delicate: empty and one-token contexts, contexts shorter
than the window, fewer eligible entries than k (-1 padding), unsorted index
sets with ineligible and out-of-range entries, two head groups (H = 128), ring
per-token caches, prefill rows with their own index sets, the overlap
eligibility rule, an explicit softmax scale, and bitwise repeatability.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B
from long_context_hybrid_02_b300 import synth
from tests._harness import assert_close, assert_lse_close, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 512
L_LONG = 6144 * 128


def _caches(Bn, L, n_cap, seed):
    s = 1 / math.sqrt(D)
    k_tok = synth.gaussian((Bn, L, D), DEV, seed, s, torch.bfloat16)
    v_tok = synth.gaussian((Bn, L, D), DEV, seed + 1, s, torch.bfloat16)
    ck = synth.gaussian((Bn, n_cap, D), DEV, seed + 2, s, torch.bfloat16)
    cv = synth.gaussian((Bn, n_cap, D), DEV, seed + 3, s, torch.bfloat16)
    return k_tok, v_tok, ck, cv


def _decode(p, q, ck, cv, n_cap, idx, k_tok, v_tok, tok_cap, ctx):
    o = torch.full((p.B, p.H, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((p.B, p.H), float("nan"), dtype=torch.float32, device=DEV)
    nb = B.ha_workspace_size(p, B.OP_DECODE, 1, n_cap, idx is not None)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV)
    B.ha_device_error(clear=True)
    B.hybrid_attn_decode(p, q, ck, cv, n_cap, idx, k_tok, v_tok, tok_cap, ctx, o, lse,
                         (ws.data_ptr(), ws.numel()))
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    return o, lse


def _check_row(o, lse, q, idx, ck, cv, K, V, t, n_win, m, scale, what, rule="disjoint"):
    """o/lse of one query row against the oracle: the row's raw index set (None:
    every eligible entry) + the window of t; the oracle ignores -1 and ineligible
    entries itself."""
    if t < 0:
        assert (np64(o) == 0).all(), what
        assert np.isneginf(np64(lse)).all(), what
        return
    if idx is not None:
        idx = np.asarray(idx.cpu() if torch.is_tensor(idx) else idx, dtype=np.int64)
    ro, rl = O.prefill_query(q, idx, ck, cv, K, V, t, n_win=n_win, m=m, scale=scale, rule=rule)
    assert_close(np64(o), ro, "bf16", what + " o")
    assert_lse_close(np64(lse), rl, "bf16", what + " lse")


def test_tc_decode_csa_ragged_contexts_and_index_sets():
    L, k, m, n_win = 8192, 512, 4, 128
    n_cap = L // m
    ctx = [0, 1, 100, 128, 140, 128 + 4 * 600, 8192]
    Bn = len(ctx)
    k_tok, v_tok, ck, cv = _caches(Bn, L, n_cap, 300)
    q = synth.gaussian((Bn, 64, D), DEV, 310, 1 / math.sqrt(D), torch.bfloat16)
    ne = [O.n_eligible(c - 1, n_win, m) if c > 0 else 0 for c in ctx]
    idx = synth.random_index_sets(Bn, 1, k, torch.tensor(ne).reshape(Bn, 1), "cpu", 7)[:, 0].clone()
    idx[6] = idx[6][torch.randperm(k, generator=torch.Generator().manual_seed(1))]  # any order
    idx[6, 10] = -1                                  # ignored
    idx[6, 11] = ne[6] + 3                           # ineligible: ignored
    idx[6, 12] = 10 ** 6                             # beyond n_cap: ignored
    idx[5, :5] = -1
    p = B.make_params(Bn, 64, D, n_win, m, k, 1, 8, B.BF16)
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    o, lse = _decode(p, q, ck, cv, n_cap, idx.to(DEV), k_tok, v_tok, L, ctx_t)
    CK, CV = np64(ck), np64(cv)
    for b, c in enumerate(ctx):
        _check_row(o[b], lse[b], np64(q[b]), idx[b], CK[b], CV[b], np64(k_tok[b]), np64(v_tok[b]),
                   c - 1, n_win, m, 1 / math.sqrt(D), f"seq {b} (ctx {c})")


def test_tc_decode_hca_two_head_groups_ring_cache():
    """H = 128 (two 64-head groups), per-token K/V in a 256-slot ring."""
    L, m, n_win, ring = 65536, 128, 128, 256
    n_cap = L // m
    ctx = [L, L - 1, L - 100, L - 128]
    Bn = len(ctx)
    k_flat, v_flat, ck, cv = _caches(Bn, L, n_cap, 320)
    k_ring = torch.empty((Bn, ring, D), dtype=torch.bfloat16, device=DEV)
    v_ring = torch.empty_like(k_ring)
    pos = torch.arange(L - ring, L, device=DEV)
    k_ring[:, pos % ring] = k_flat[:, L - ring:]
    v_ring[:, pos % ring] = v_flat[:, L - ring:]
    q = synth.gaussian((Bn, 128, D), DEV, 330, 1 / math.sqrt(D), torch.bfloat16)
    p = B.make_params(Bn, 128, D, n_win, m, 1, 1, 8, B.BF16)
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    o, lse = _decode(p, q, ck, cv, n_cap, None, k_ring, v_ring, ring, ctx_t)
    CK, CV = np64(ck), np64(cv)
    for b, c in enumerate(ctx):
        _check_row(o[b], lse[b], np64(q[b]), None, CK[b], CV[b], np64(k_flat[b]),
                   np64(v_flat[b]), c - 1, n_win, m, 1 / math.sqrt(D), f"seq {b} (ctx {c})")


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_tc_prefill_rows_with_own_sets_and_windows(kind):
    """12 queries per sequence at scattered positions (not block-aligned), each with
    its own index set (CSA) and causal window."""
    L, n_win = 16384, 128
    m = 4 if kind == "csa" else 128
    k = 512 if kind == "csa" else 1
    n_cap = L // m
    Bn, Tq = 2, 12
    k_tok, v_tok, ck, cv = _caches(Bn, L, n_cap, 340)
    rng = np.random.default_rng(4)
    pos = np.sort(rng.integers(0, L, (Bn, Tq)), axis=1)
    pos[0, :3] = [0, 127, 130]
    q_pos = torch.tensor(pos, dtype=torch.int32, device=DEV)
    q = synth.gaussian((Bn, Tq, 64, D), DEV, 350, 1 / math.sqrt(D), torch.bfloat16)
    ne = torch.tensor([[O.n_eligible(int(t), n_win, m) for t in row] for row in pos])
    idx = None
    if kind == "csa":
        idx = synth.random_index_sets(Bn, Tq, k, ne, DEV, 9)
    p = B.make_params(Bn, 64, D, n_win, m, k, 1, 8, B.BF16)
    o = torch.full((Bn, Tq, 64, D), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((Bn, Tq, 64), float("nan"), dtype=torch.float32, device=DEV)
    nb = B.ha_workspace_size(p, B.OP_PREFILL, Tq, n_cap, idx is not None)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV)
    B.ha_device_error(clear=True)
    B.hybrid_attn_prefill(p, q, q_pos, Tq, ck, cv, n_cap, idx, k_tok, v_tok, L, o, lse,
                          (ws.data_ptr(), ws.numel()))
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    CK, CV = np64(ck), np64(cv)
    for b in range(Bn):
        K, V = np64(k_tok[b]), np64(v_tok[b])
        for i in range(Tq):
            t = int(pos[b, i])
            _check_row(o[b, i], lse[b, i], np64(q[b, i]), idx[b, i] if kind == "csa" else None,
                       CK[b], CV[b], K, V, t, n_win, m,
                       1 / math.sqrt(D), f"[{b},{i}] t={t}")


def test_tc_decode_overlap_rule_and_explicit_scale():
    L, k, m, n_win = 4096, 512, 4, 128
    n_cap = L // m
    ctx = [4096, 777, 130]
    Bn = len(ctx)
    k_tok, v_tok, ck, cv = _caches(Bn, L, n_cap, 360)
    q = synth.gaussian((Bn, 64, D), DEV, 370, 1 / math.sqrt(D), torch.bfloat16)
    ne = [O.n_eligible(c - 1, n_win, m, "overlap") for c in ctx]
    idx = synth.random_index_sets(Bn, 1, k, torch.tensor(ne).reshape(Bn, 1), DEV, 11)[:, 0].contiguous()
    scale = 0.07
    p = B.make_params(Bn, 64, D, n_win, m, k, 1, 8, B.BF16, B.ELIG_OVERLAP, scale)
    o, lse = _decode(p, q, ck, cv, n_cap, idx, k_tok, v_tok, L,
                     torch.tensor(ctx, dtype=torch.int32, device=DEV))
    CK, CV = np64(ck), np64(cv)
    for b, c in enumerate(ctx):
        _check_row(o[b], lse[b], np64(q[b]), idx[b], CK[b], CV[b], np64(k_tok[b]), np64(v_tok[b]),
                   c - 1, n_win, m, scale, f"seq {b}", rule="overlap")


def test_tc_decode_bitwise_repeatable_and_position_invariant():
    """Fixed reduction orders: two runs give the same bits, and the same sequence
    at two batch positions of one launch gives the same bits."""
    L, k, m, n_win = 8192, 512, 4, 128
    n_cap = L // m
    k_tok, v_tok, ck, cv = _caches(1, L, n_cap, 380)
    rep = lambda t: t.expand(3, *t.shape[1:]).contiguous()
    k_tok, v_tok, ck, cv = rep(k_tok), rep(v_tok), rep(ck), rep(cv)
    q = rep(synth.gaussian((1, 64, D), DEV, 390, 1 / math.sqrt(D), torch.bfloat16))
    ne = O.n_eligible(L - 1, n_win, m)
    idx = rep(synth.random_index_sets(1, 1, k, torch.tensor([[ne]]), DEV, 13)[:, 0].contiguous())
    p = B.make_params(3, 64, D, n_win, m, k, 1, 8, B.BF16)
    ctx = torch.full((3,), L, dtype=torch.int32, device=DEV)
    o1, l1 = _decode(p, q, ck, cv, n_cap, idx, k_tok, v_tok, L, ctx)
    o2, l2 = _decode(p, q, ck, cv, n_cap, idx, k_tok, v_tok, L, ctx)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1[0], o1[2]) and torch.equal(l1[0], l1[2])


@pytest.mark.parametrize("ctx_off", [(0, 77), (0, 77, L_LONG - 200, L_LONG)])
def test_tc_decode_hca_long_rows_in_several_cluster_groups(ctx_off):
    """Up to 6,144 + 128 keys per row and few rows: every row's keys are cut into
    many splits whose float32 results are merged by a second launch; a 200-token
    and an empty context leave whole splits without keys."""
    m, n_win, ring = 128, 128, 256
    n_cap = 6144
    L = n_cap * m
    ctx = [L - off for off in ctx_off]
    Bn = len(ctx)
    s = 1 / math.sqrt(D)
    ck = synth.gaussian((Bn, n_cap, D), DEV, 400, s, torch.bfloat16)
    cv = synth.gaussian((Bn, n_cap, D), DEV, 401, s, torch.bfloat16)
    win_k = synth.gaussian((Bn, ring, D), DEV, 402, s, torch.bfloat16)   # positions L-256 .. L-1
    win_v = synth.gaussian((Bn, ring, D), DEV, 403, s, torch.bfloat16)
    k_ring = torch.empty_like(win_k)
    v_ring = torch.empty_like(win_v)
    pos = torch.arange(L - ring, L, device=DEV)
    k_ring[:, pos % ring] = win_k
    v_ring[:, pos % ring] = win_v
    q = synth.gaussian((Bn, 64, D), DEV, 404, s, torch.bfloat16)
    p = B.make_params(Bn, 64, D, n_win, m, 1, 1, 8, B.BF16)
    o, lse = _decode(p, q, ck, cv, n_cap, None, k_ring, v_ring, ring,
                     torch.tensor(ctx, dtype=torch.int32, device=DEV))
    CK, CV = np64(ck), np64(cv)
    for b, c in enumerate(ctx):
        t = c - 1
        if t < 0:
            assert (np64(o[b]) == 0).all() and np.isneginf(np64(lse[b])).all()
            continue
        ne = O.n_eligible(t, n_win, m)
        win = O.window_positions(t, n_win)
        keys = np.concatenate([CK[b, :ne], np64(k_ring[b])[win % ring]])    # the slots read
        vals = np.concatenate([CV[b, :ne], np64(v_ring[b])[win % ring]])
        ro, rl = O.attend(np64(q[b]), keys, vals, 1 / math.sqrt(D))
        assert_close(np64(o[b]), ro, "bf16", f"o[{b}]")
        assert_lse_close(np64(lse[b]), rl, "bf16", f"lse[{b}]")


@pytest.mark.parametrize("Bn,k", [(48, 512), (32, 512), (20, 512), (32, 200)])
def test_tc_decode_split_tails_of_every_size(Bn, k):
    """Batch sizes that give 3, 4 and 7 splits per row: the last tile of a split
    holds 128, 96, 64, 40 or 32 keys, so every compact tail size (32, 64 and 128
    rows per stage set) meets real keys."""
    L, m, n_win = 4096, 4, 128
    n_cap = L // m
    k_tok, v_tok, ck, cv = _caches(Bn, L, n_cap, 400 + Bn + k)
    q = synth.gaussian((Bn, 64, D), DEV, 410 + Bn, 1 / math.sqrt(D), torch.bfloat16)
    ne = O.n_eligible(L - 1, n_win, m)
    idx = synth.random_index_sets(Bn, 1, k, torch.full((Bn, 1), ne), "cpu", 9)[:, 0].clone()
    p = B.make_params(Bn, 64, D, n_win, m, k, 1, 8, B.BF16)
    ctx_t = torch.full((Bn,), L, dtype=torch.int32, device=DEV)
    o, lse = _decode(p, q, ck, cv, n_cap, idx.to(DEV), k_tok, v_tok, L, ctx_t)
    CK, CV = np64(ck), np64(cv)
    for b in range(Bn):
        _check_row(o[b], lse[b], np64(q[b]), idx[b], CK[b], CV[b], np64(k_tok[b]), np64(v_tok[b]),
                   L - 1, n_win, m, 1 / math.sqrt(D), f"seq {b}")

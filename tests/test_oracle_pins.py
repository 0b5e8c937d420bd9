"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to a hand-derived worked example
(tests/golden/worked_examples.json), a closed form, an invariant, a textbook
routine (torch's float64 scaled_dot_product_attention, heapq, math.fsum) or brute
force on tiny inputs.  The last group plants plausible mistakes into the oracle
(monkeypatched, on the CPU) and checks that a pin catches each of them.
"""
import heapq
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import hybrid_attention as O

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")))


def sdpa64(q, keys, values, scale):
    """Textbook attention of H queries over n keys (torch, float64, no mask)."""
    qt = torch.tensor(q, dtype=torch.float64)[None, :, None, :]        # [1, H, 1, d]
    kt = torch.tensor(keys, dtype=torch.float64)[None, None].expand(1, q.shape[0], -1, -1)
    vt = torch.tensor(values, dtype=torch.float64)[None, None].expand(1, q.shape[0], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[0, :, 0, :].numpy()


# ----------------------------------------------------------------- storage rounding
def test_bf16_rounding_ties_and_exact_values():
    g = GOLD["bf16_rounding"]
    got = O.round_to_bf16(np.array(g["inputs"]))
    assert got.tolist() == g["expected"]


def test_bf16_rounding_matches_torch_on_float32_values():
    # float32-representable inputs round once in both routes, so they must agree bit for bit
    rng = np.random.default_rng(1)
    x32 = (rng.standard_normal(200000) * np.exp(rng.uniform(-20, 20, 200000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_to_bf16(x32.astype(np.float64)), ref)


# ----------------------------------------------------------------- compressor
def test_compress_worked_example():
    g = GOLD["compress_block"]
    out = O.compress_block(np.array(g["rows"], float), np.log(np.array(g["gate_exp"])))
    np.testing.assert_allclose(out, g["expected"], rtol=0, atol=1e-14)


def test_gate_softmax_sums_to_one():
    rng = np.random.default_rng(2)
    for m in (1, 4, 128):
        for _ in range(20):
            a = O.gate_softmax(rng.standard_normal(m) * 5)
            assert abs(a.sum() - 1.0) < 1e-12 and (a >= 0).all()


def test_compress_constant_block_gives_constant():
    rng = np.random.default_rng(3)
    for m in (4, 128):
        row = rng.standard_normal(16)
        X = np.tile(row, (3 * m, 1))
        out = O.compress(X, rng.standard_normal(3 * m) * 3, m, 0, 3)
        np.testing.assert_allclose(out, np.tile(row, (3, 1)), rtol=1e-13, atol=1e-14)


def test_compress_equal_gates_gives_mean_and_dominant_gate_gives_token():
    rng = np.random.default_rng(4)
    m, d = 4, 8
    X = rng.standard_normal((2 * m, d))
    eq = O.compress(X, np.full(2 * m, 0.7), m, 0, 2)
    np.testing.assert_allclose(eq, X.reshape(2, m, d).mean(axis=1), rtol=1e-13, atol=1e-15)
    g = rng.standard_normal(2 * m)
    g[2] += 60.0          # token 2 of block 0
    g[7] += 60.0          # token 3 of block 1
    dom = O.compress(X, g, m, 0, 2)
    np.testing.assert_allclose(dom, X[[2, 7]], rtol=1e-12, atol=1e-12)


def test_compress_is_convex_and_identity_for_m1():
    rng = np.random.default_rng(5)
    m = 128
    X = rng.standard_normal((2 * m, 32))
    out = O.compress(X, rng.standard_normal(2 * m), m, 0, 2)
    blocks = X.reshape(2, m, 32)
    assert (out <= blocks.max(axis=1) + 1e-12).all() and (out >= blocks.min(axis=1) - 1e-12).all()
    np.testing.assert_array_equal(O.compress(X, rng.standard_normal(2 * m), 1, 5, 7), X[5:12])


def test_compress_brute_force_tiny():
    rng = np.random.default_rng(6)
    m, d = 4, 3
    X = rng.standard_normal((3 * m, d))
    g = rng.standard_normal(3 * m)
    out = O.compress(X, g, m, 1, 2)
    for b, j in enumerate((1, 2)):
        ws = [math.exp(g[j * m + i]) for i in range(m)]
        tot = math.fsum(ws)
        for c in range(d):
            ref = math.fsum(ws[i] / tot * X[j * m + i, c] for i in range(m))
            assert abs(out[b, c] - ref) < 1e-14


def test_compress_rounds_to_the_cache_storage_type():
    """The compressed cache holds entries in its storage type: the bf16 result is
    torch's float64 -> bfloat16 cast of the fp64 result (on the bf16 grid), the
    fp32 result its float32 cast."""
    rng = np.random.default_rng(14)
    X, g = rng.standard_normal((64, 40)) / 7, rng.standard_normal(64)
    exact = O.compress(X, g, 4, 0, 16)
    for storage, dt in (("bf16", torch.bfloat16), ("f32", torch.float32)):
        got = O.compress(X, g, 4, 0, 16, storage)
        ref = torch.tensor(exact, dtype=torch.float64).to(dt).double().numpy()
        np.testing.assert_array_equal(got, ref)
    assert not np.array_equal(O.compress(X, g, 4, 0, 16, "bf16"), exact)


def test_compress_rejects_incomplete_block():
    with pytest.raises(ValueError):
        O.compress(np.zeros((10, 2)), np.zeros(10), 4, 2, 1)


# ----------------------------------------------------------------- eligibility / window
def test_eligibility_by_enumeration():
    # brute force: a block is eligible (disjoint rule) iff its last token precedes the window
    for n_win in (1, 4, 128):
        for m in (1, 4, 128):
            for t in list(range(0, 400, 7)) + [n_win - 1, n_win, n_win + m - 1, n_win + m]:
                win_lo = max(0, t - n_win + 1)
                ref = sum(1 for j in range(t + 2) if (j + 1) * m - 1 < win_lo)
                assert O.n_eligible(t, n_win, m) == ref
                assert O.n_eligible(t, n_win, m, "overlap") == sum(
                    1 for j in range(t + 2) if (j + 1) * m - 1 <= t)
                w = O.window_positions(t, n_win)
                assert len(w) == min(n_win, t + 1) and w[-1] == t


# ----------------------------------------------------------------- indexer
def test_index_scores_worked_example():
    g = GOLD["index_scores"]
    s = O.index_scores(np.array(g["qI"], float), np.array(g["w"]), np.array(g["cI"], float))
    assert s.tolist() == g["expected_scores"]
    assert O.topk_select(s, 2).tolist() == g["expected_top2"]
    assert O.topk_select(s, 3).tolist() == g["expected_top3"]
    assert O.topk_select(s, 6).tolist() == g["expected_top6"]


def test_index_scores_single_head_and_brute_force():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((1, 16))
    c = rng.standard_normal((40, 16))
    s = O.index_scores(q, np.ones(1), c)
    ref = [max(0.0, math.fsum(q[0, i] * c[j, i] for i in range(16))) for j in range(40)]
    np.testing.assert_allclose(s, ref, rtol=1e-13, atol=1e-14)
    H = 3
    q = rng.standard_normal((H, 8))
    w = rng.uniform(0, 1, H)
    c = rng.standard_normal((25, 8))
    s = O.index_scores(q, w, c)
    for j in range(25):
        ref = math.fsum(w[h] * max(0.0, math.fsum(q[h, i] * c[j, i] for i in range(8)))
                        for h in range(H))
        assert abs(s[j] - ref) < 1e-13


def test_index_scores_negative_dots_and_linearity():
    rng = np.random.default_rng(8)
    q = np.abs(rng.standard_normal((4, 8)))
    c = -np.abs(rng.standard_normal((10, 8)))
    assert (O.index_scores(q, np.ones(4), c) == 0).all()
    q = rng.standard_normal((4, 8))
    c = rng.standard_normal((10, 8))
    w1, w2 = rng.uniform(0, 1, 4), rng.uniform(0, 1, 4)
    np.testing.assert_allclose(O.index_scores(q, w1 + 2 * w2, c),
                               O.index_scores(q, w1, c) + 2 * O.index_scores(q, w2, c),
                               rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------- top-k
def test_topk_matches_heap_selection_with_ties_and_nan():
    rng = np.random.default_rng(9)
    for n, k in ((1, 1), (7, 3), (50, 50), (300, 16), (6000, 512)):
        s = np.round(rng.standard_normal(n), 1)       # many exact ties
        s[rng.integers(0, n, max(1, n // 50))] = np.nan
        ref = heapq.nsmallest(k, range(n), key=lambda j: (
            math.inf if math.isnan(s[j]) else -s[j], j))
        got = O.topk_select(s, k)
        assert got[got >= 0].tolist() == sorted(ref)


def test_topk_signed_zeros_are_one_score():
    # -0.0 == +0.0 as numbers, so they tie and the smaller index wins
    s = np.array([-0.0, 0.0, -0.0, 0.0, -1.0])
    assert O.topk_select(s, 2).tolist() == [0, 1]
    assert O.topk_select(np.array([0.0, -0.0, 0.0]), 1).tolist() == [0]


def test_topk_pads_when_fewer_than_k_and_handles_empty():
    assert O.topk_select(np.array([0.5, -1.0, 2.0]), 5).tolist() == [0, 1, 2, -1, -1]
    assert O.topk_select(np.array([]), 3).tolist() == [-1, -1, -1]


def test_topk_equivariant_under_permutation():
    rng = np.random.default_rng(10)
    s = rng.standard_normal(1000)
    perm = rng.permutation(1000)
    a = O.topk_select(s, 64)
    b = O.topk_select(s[perm], 64)
    assert sorted(perm[b].tolist()) == a.tolist()


# ----------------------------------------------------------------- attention
def test_attend_worked_example():
    g = GOLD["attend"]
    keys = np.zeros((2, 4))
    keys[g["k_ln3_at"][0], g["k_ln3_at"][1]] = math.log(3.0)
    o, lse = O.attend(np.array(g["q"], float), keys, np.array(g["values"], float), g["scale"])
    np.testing.assert_allclose(o, g["expected_o"], rtol=0, atol=1e-15)
    assert abs(math.exp(lse[0]) - g["expected_lse_exp"]) < 1e-13


def test_attend_matches_textbook_sdpa():
    rng = np.random.default_rng(11)
    q, k, v = rng.standard_normal((8, 64)), rng.standard_normal((100, 64)), rng.standard_normal((100, 48))
    o, lse = O.attend(q, k, v, 0.125)
    np.testing.assert_allclose(o, sdpa64(q, k, v, 0.125), rtol=1e-12, atol=1e-13)
    ref_lse = [math.log(math.fsum(math.exp(0.125 * float(q[h] @ k[j])) for j in range(100)))
               for h in range(8)]
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13)


def test_attend_rows_sum_to_one_single_key_and_empty():
    rng = np.random.default_rng(12)
    q, k = rng.standard_normal((5, 16)), rng.standard_normal((30, 16))
    p, _ = O.attend(q, k, np.eye(30), 0.3)          # one-hot values expose p itself
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (p >= 0).all()
    v1 = rng.standard_normal((1, 16))
    o, lse = O.attend(q, k[:1], v1, 0.3)
    np.testing.assert_allclose(o, np.repeat(v1, 5, axis=0), rtol=1e-14)
    np.testing.assert_allclose(lse, 0.3 * q @ k[0], rtol=1e-14)
    o, lse = O.attend(q, np.zeros((0, 16)), np.zeros((0, 16)), 0.3)
    assert (o == 0).all() and np.isneginf(lse).all()


def test_merge_partials_equals_joint_attention():
    rng = np.random.default_rng(13)
    q, k, v = rng.standard_normal((4, 32)), rng.standard_normal((90, 32)), rng.standard_normal((90, 32))
    ref_o, ref_l = O.attend(q, k, v, 0.2)
    cuts = [0, 7, 7, 40, 90]                         # includes an empty part
    parts = [O.attend(q, k[a:b], v[a:b], 0.2) for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = O.merge_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, ref_l, rtol=1e-13)


# ----------------------------------------------------------------- layer-level invariants
def _tokens(rng, L, d):
    return rng.standard_normal((L, d)) / math.sqrt(d), rng.standard_normal((L, d)) / math.sqrt(d)


@pytest.mark.parametrize("t", [0, 5, 127, 128, 129, 300, 511])
def test_csa_with_m1_and_large_k_is_full_causal_attention(t):
    """m = 1 and k >= #entries: every earlier token is seen exactly once."""
    rng = np.random.default_rng(100 + t)
    L, d, H, n_win = 512, 32, 4, 128
    K, V = _tokens(rng, L, d)
    gate = rng.standard_normal(L)
    ck, cv = O.compress(K, gate, 1, 0, L), O.compress(V, gate, 1, 0, L)
    qI, w = rng.standard_normal((2, 8)), rng.uniform(0, 1, 2)
    cI = O.compress(rng.standard_normal((L, 8)), gate, 1, 0, L)
    q = rng.standard_normal((H, d))
    o, lse, idx, _ = O.csa_decode(q, qI, w, ck, cv, cI, K, V, t, n_win=n_win, m=1, k=L,
                                  scale=d ** -0.5)
    np.testing.assert_allclose(o, sdpa64(q, K[:t + 1], V[:t + 1], d ** -0.5), rtol=1e-11, atol=1e-13)


@pytest.mark.parametrize("t", [0, 60, 127, 128 + 126])
def test_hca_reduces_to_swa_when_no_block_is_eligible(t):
    """Context <= n_win (or < n_win + m'): only the window is attended."""
    rng = np.random.default_rng(200 + t)
    L, d, H, n_win, m = 256, 16, 3, 128, 128
    K, V = _tokens(rng, L, d)
    gate = rng.standard_normal(L)
    ck, cv = O.compress(K, gate, m, 0, 2), O.compress(V, gate, m, 0, 2)
    q = rng.standard_normal((H, d))
    o, _ = O.hca_decode(q, ck, cv, K, V, t, n_win=n_win, m=m, scale=0.25)
    lo = max(0, t - n_win + 1)
    np.testing.assert_allclose(o, sdpa64(q, K[lo:t + 1], V[lo:t + 1], 0.25), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("kind,m,t", [("hca", 128, 1023), ("hca", 128, 700), ("csa", 4, 1023),
                                      ("csa", 4, 301), ("hca", 4, 150)])
def test_layer_with_blockwise_constant_kv_is_attention_over_block_rows(kind, m, t):
    """If K, V are constant inside every block, an entry equals its block's row, so the
    layer is plain attention over [eligible block rows] + [window tokens], with the
    eligible blocks counted here by enumeration."""
    rng = np.random.default_rng(300 + t + m)
    d, H, n_win, L = 32, 4, 128, 1024
    nb = L // m
    Kb, Vb = _tokens(rng, nb, d)
    K, V = np.repeat(Kb, m, axis=0), np.repeat(Vb, m, axis=0)
    # the window keeps its own (distinct) tokens
    Kw, Vw = _tokens(rng, L, d)
    lo = max(0, t - n_win + 1)
    K[lo:t + 1], V[lo:t + 1] = Kw[lo:t + 1], Vw[lo:t + 1]
    gate = rng.standard_normal(L) * 2
    elig = [j for j in range(nb) if (j + 1) * m - 1 < lo]
    # compressed caches of blocks overlapping the window are never read; compress from
    # the block-constant rows so that every entry equals its block row
    ck = O.compress(np.repeat(Kb, m, axis=0), gate, m, 0, nb)
    cv = O.compress(np.repeat(Vb, m, axis=0), gate, m, 0, nb)
    q = rng.standard_normal((H, d))
    keys = np.concatenate([Kb[elig], K[lo:t + 1]])
    vals = np.concatenate([Vb[elig], V[lo:t + 1]])
    ref = sdpa64(q, keys, vals, d ** -0.5)
    if kind == "hca":
        o, _ = O.hca_decode(q, ck, cv, K, V, t, n_win=n_win, m=m, scale=d ** -0.5)
    else:
        qI, w = rng.standard_normal((2, 8)), rng.uniform(0, 1, 2)
        cI = rng.standard_normal((nb, 8))
        o, _, idx, _ = O.csa_decode(q, qI, w, ck, cv, cI, K, V, t, n_win=n_win, m=m, k=nb,
                                    scale=d ** -0.5)
        assert idx[idx >= 0].tolist() == elig
    np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-14)


def test_csa_selects_exactly_the_topk_entries():
    """With a large gap between k planted entries and the rest, CSA attends exactly to
    the planted entries plus the window (checked against attention over that set)."""
    rng = np.random.default_rng(400)
    L, d, H, m, n_win, k = 2048, 16, 2, 4, 128, 8
    nb = L // m
    K, V = _tokens(rng, L, d)
    gate = rng.standard_normal(L)
    ck, cv = O.compress(K, gate, m, 0, nb), O.compress(V, gate, m, 0, nb)
    qI = rng.standard_normal((2, 8))
    w = np.array([1.0, 0.5])
    cI = rng.standard_normal((nb, 8)) * 0.01
    planted = np.sort(rng.choice(O.n_eligible(L - 1, n_win, m), k, replace=False))
    cI[planted] = qI[0] * 10.0
    q = rng.standard_normal((H, d))
    t = L - 1
    o, _, idx, _ = O.csa_decode(q, qI, w, ck, cv, cI, K, V, t, n_win=n_win, m=m, k=k, scale=0.25)
    assert idx.tolist() == planted.tolist()
    keys = np.concatenate([ck[planted], K[t - n_win + 1:]])
    vals = np.concatenate([cv[planted], V[t - n_win + 1:]])
    np.testing.assert_allclose(o, sdpa64(q, keys, vals, 0.25), rtol=1e-12, atol=1e-14)


def test_prefill_query_equals_decode_at_that_position():
    rng = np.random.default_rng(500)
    L, d, H, m, n_win = 700, 16, 2, 128, 128
    K, V = _tokens(rng, L, d)
    gate = rng.standard_normal(L)
    nb = L // m
    ck, cv = O.compress(K, gate, m, 0, nb), O.compress(V, gate, m, 0, nb)
    q = rng.standard_normal((H, d))
    for t in (0, 200, 255, 256, 699):
        a, la = O.prefill_query(q, None, ck, cv, K, V, t, n_win=n_win, m=m, scale=0.3)
        b, lb = O.hca_decode(q, ck, cv, K[:t + 1], V[:t + 1], t, n_win=n_win, m=m, scale=0.3)
        np.testing.assert_allclose(a, b, rtol=1e-14)


def _eligible_by_enumeration(t, n_win, m, n_cap):
    """Entries whose whole block ends before the window of t, listed one by one."""
    lo = max(0, t - n_win + 1)
    return [j for j in range(n_cap) if (j + 1) * m - 1 < lo]


@pytest.mark.parametrize("t", [0, 130, 131, 300, 599])
def test_prefill_query_with_a_selection_attends_its_eligible_entries_and_the_window(t):
    """A query with a given selection (unsorted, -1 padded, with entries beyond the
    eligible blocks, beyond the cache and listed twice) attends exactly to the
    listed eligible entries, each as often as listed, plus its window: textbook
    float64 attention over that key list, with eligibility enumerated here."""
    rng = np.random.default_rng(600 + t)
    L, d, H, m, n_win = 600, 16, 3, 4, 128
    K, V = _tokens(rng, L, d)
    for n_cap in (L // m, 20):                      # 20 rows: a cache shorter than n_elig
        ck, cv = _tokens(rng, n_cap, d)
        elig = _eligible_by_enumeration(t, n_win, m, n_cap)
        chosen = list(rng.permutation(elig)[:7]) if elig else []
        if chosen:
            chosen.append(chosen[0])                # listed twice
        over = [n_cap - 1 + 5, L // m + 3, 10 ** 6]  # never eligible for this cache
        if len(elig) < n_cap:
            over.append(len(elig))                  # first block overlapping the window
        idx = np.array(chosen + over + [-1, -1, -7], dtype=np.int64)[rng.permutation(len(chosen) + len(over) + 3)]
        q = rng.standard_normal((H, d))
        keep = [int(j) for j in idx if int(j) in set(elig)]
        lo = max(0, t - n_win + 1)
        keys = np.concatenate([ck[keep].reshape(-1, d), K[lo:t + 1]])
        vals = np.concatenate([cv[keep].reshape(-1, d), V[lo:t + 1]])
        o, lse = O.prefill_query(q, idx, ck, cv, K, V, t, n_win=n_win, m=m, scale=d ** -0.5)
        np.testing.assert_allclose(o, sdpa64(q, keys, vals, d ** -0.5), rtol=1e-12, atol=1e-14)
        # the same query given only its window's per-token rows (row 0 = position lo)
        o2, lse2 = O.prefill_query(q, idx, ck, cv, K[lo:t + 1], V[lo:t + 1], t, n_win=n_win, m=m,
                                   scale=d ** -0.5, tok_base=lo)
        assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
        z = (d ** -0.5) * q @ keys.T
        np.testing.assert_allclose(lse, [math.log(math.fsum(np.exp(r))) for r in z], rtol=1e-13)


# ----------------------------------------------------------------- planted mistakes
def test_pins_catch_an_off_by_one_eligibility(monkeypatch):
    good = O.n_eligible
    monkeypatch.setattr(O, "n_eligible", lambda t, n_win, m, rule="disjoint": good(t + 1, n_win, m, rule))
    with pytest.raises(AssertionError):
        test_csa_with_m1_and_large_k_is_full_causal_attention(300)


def test_pins_catch_a_wrong_window(monkeypatch):
    monkeypatch.setattr(O, "window_positions", lambda t, n_win: np.arange(max(0, t - n_win), t + 1))
    with pytest.raises(AssertionError):
        test_hca_reduces_to_swa_when_no_block_is_eligible(254)


def test_pins_catch_a_transposed_gate_weighting(monkeypatch):
    monkeypatch.setattr(O, "gate_softmax", lambda g: (lambda e: e[::-1] / e.sum())(
        np.exp(np.asarray(g, float) - np.max(g))))
    with pytest.raises(AssertionError):
        test_compress_worked_example()


def test_pins_catch_a_dropped_relu(monkeypatch):
    monkeypatch.setattr(O, "index_scores", lambda qI, w, cI: (np.asarray(cI, float) @ np.asarray(qI, float).T) @ np.asarray(w, float))
    with pytest.raises(AssertionError):
        test_index_scores_worked_example()


def test_pins_catch_a_squared_softmax_scale(monkeypatch):
    good = O.attend
    monkeypatch.setattr(O, "attend", lambda q, k, v, scale: good(q, k, v, scale * scale))
    with pytest.raises(AssertionError):
        test_attend_matches_textbook_sdpa()


def _bad_topk(larger_index_first: bool, sort_output: bool):
    def topk(scores, k):
        s = np.asarray(scores, dtype=np.float64).copy()
        s[np.isnan(s)] = -np.inf
        n = s.shape[0]
        tie = -np.arange(n) if larger_index_first else np.arange(n)
        order = np.lexsort((tie, -s))[:min(k, n)]
        out = np.full(k, -1, dtype=np.int64)
        out[:order.size] = np.sort(order) if sort_output else order
        return out
    return topk


def test_pins_catch_ties_broken_toward_the_larger_index(monkeypatch):
    monkeypatch.setattr(O, "topk_select", _bad_topk(larger_index_first=True, sort_output=True))
    with pytest.raises(AssertionError):
        test_topk_matches_heap_selection_with_ties_and_nan()


def test_pins_catch_a_selection_left_in_score_order(monkeypatch):
    monkeypatch.setattr(O, "topk_select", _bad_topk(larger_index_first=False, sort_output=False))
    with pytest.raises(AssertionError):
        test_topk_matches_heap_selection_with_ties_and_nan()


def test_pins_catch_a_merge_that_ignores_the_lse_weights(monkeypatch):
    monkeypatch.setattr(O, "merge_partials", lambda o, lse: (np.asarray(o).mean(axis=0),
                                                              np.asarray(lse).max(axis=0)))
    with pytest.raises(AssertionError):
        test_merge_partials_equals_joint_attention()


def test_pins_catch_separate_softmaxes_for_window_and_entries(monkeypatch):
    good_attend, good_ne = O.attend, O.n_eligible

    def two_softmaxes(q, ck, cv, k_tok, v_tok, t, *, n_win, m, scale, rule="disjoint"):
        ne = good_ne(t, n_win, m, rule)
        win = O.window_positions(t, n_win)
        ow, lw = good_attend(q, k_tok[win], v_tok[win], scale)
        if ne == 0:
            return ow, lw
        oc, lc = good_attend(q, ck[:ne], cv[:ne], scale)
        return (ow + oc) / 2, np.logaddexp(lw, lc)

    monkeypatch.setattr(O, "hca_decode", two_softmaxes)
    with pytest.raises(AssertionError):
        test_layer_with_blockwise_constant_kv_is_attention_over_block_rows("hca", 128, 1023)


def test_pins_catch_bf16_by_truncation(monkeypatch):
    def truncate(x):
        a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
        return (a.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)
    monkeypatch.setattr(O, "round_to_bf16", truncate)
    with pytest.raises(AssertionError):
        test_bf16_rounding_ties_and_exact_values()


def test_pins_catch_an_unrounded_cache(monkeypatch):
    monkeypatch.setattr(O, "round_to_storage", lambda x, storage: np.asarray(x, dtype=np.float64))
    with pytest.raises(AssertionError):
        test_compress_rounds_to_the_cache_storage_type()


def _query_with(keep):
    """prefill_query whose selection filter is `keep(idx, ne, n_cap)` (a planted mistake)."""
    def prefill_query(q, idx, ck, cv, k_tok, v_tok, t, *, n_win, m, scale, rule="disjoint"):
        n_cap = np.asarray(ck).shape[0]
        ne = min(O.n_eligible(t, n_win, m, rule), n_cap)
        idx = np.asarray(idx, dtype=np.int64)
        sel = idx[keep(idx, ne, n_cap)]
        keys = np.concatenate([np.asarray(ck)[sel], np.asarray(k_tok)[O.window_positions(t, n_win)]])
        vals = np.concatenate([np.asarray(cv)[sel], np.asarray(v_tok)[O.window_positions(t, n_win)]])
        return O.attend(q, keys, vals, scale)
    return prefill_query


def test_pins_catch_a_selection_whose_padding_is_not_filtered(monkeypatch):
    # -1 kept: numpy reads it as the cache's last row
    monkeypatch.setattr(O, "prefill_query", _query_with(lambda i, ne, n: (i < ne)))
    with pytest.raises(AssertionError):
        test_prefill_query_with_a_selection_attends_its_eligible_entries_and_the_window(300)


def test_pins_catch_a_selection_that_keeps_ineligible_entries(monkeypatch):
    monkeypatch.setattr(O, "prefill_query", _query_with(lambda i, ne, n: (i >= 0) & (i < n)))
    with pytest.raises(AssertionError):
        test_prefill_query_with_a_selection_attends_its_eligible_entries_and_the_window(300)


def test_pins_catch_a_selection_that_drops_repeated_entries(monkeypatch):
    monkeypatch.setattr(O, "prefill_query", _query_with(
        lambda i, ne, n: ((i >= 0) & (i < ne)) & (np.unique(i, return_index=True)[1][
            np.searchsorted(np.unique(i), i)] == np.arange(i.size))))
    with pytest.raises(AssertionError):
        test_prefill_query_with_a_selection_attends_its_eligible_entries_and_the_window(300)


def test_oracle_package_exports():
    for name in O.__all__:
        assert getattr(oracle, name) is getattr(O, name)

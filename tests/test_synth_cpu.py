"""CPU checks of the seeded input generators, the one module that both the CUDA
path and the oracle read their inputs from.  It computes none of the method, so
these tests pin only what the inputs are meant to be: the same draws for the
same seed, the documented shapes, types and scales, rotary embedding as a
rotation of each interleaved pair, the planted component of the long-context
workload, and well-formed stand-in index sets.
"""
import math

import numpy as np
import pytest
import torch

from long_context_hybrid_02_b300 import synth


def small(kind="csa", **kw):
    base = synth.WORKLOADS["tiny_" + kind]
    return base.scaled(**kw)


@pytest.mark.parametrize("kind", ["csa", "hca"])
def test_same_seed_same_draws_other_seed_other_draws(kind):
    w = small(kind, L=2048)
    a, b = synth.make_tokens(w, "cpu"), synth.make_tokens(w, "cpu")
    qa, qb = synth.make_queries(w, "cpu"), synth.make_queries(w, "cpu")
    for name in a:
        assert torch.equal(a[name], b[name]), name
    for name in qa:
        assert torch.equal(qa[name], qb[name]), name
    c = synth.make_tokens(w.scaled(seed=1), "cpu")
    for name in a:
        assert not torch.equal(a[name], c[name]), name
    # every tensor is drawn from its own stream: K and V of one seed differ
    assert not torch.equal(a["k_tok"], a["v_tok"])


@pytest.mark.parametrize("kind,dtype", [("csa", "f32"), ("csa", "bf16"), ("hca", "bf16")])
def test_shapes_and_types(kind, dtype):
    w = small(kind, B=2, L=1536, dtype=dtype, Tq=3)
    tok = synth.make_tokens(w, "cpu")
    qry = synth.make_queries(w, "cpu")
    dt = torch.float32 if dtype == "f32" else torch.bfloat16
    assert tok["k_tok"].shape == (2, 1536, w.d) and tok["k_tok"].dtype == dt
    assert tok["v_tok"].shape == (2, 1536, w.d) and tok["v_tok"].dtype == dt
    assert tok["gate"].shape == (2, 1536) and tok["gate"].dtype == torch.float32
    assert qry["q"].shape == (2, 3, w.H, w.d) and qry["q"].dtype == dt
    assert qry["q"].is_contiguous()
    assert torch.equal(qry["ctx_len"], torch.full((2,), 1536, dtype=torch.int32))
    assert torch.equal(qry["q_pos"], torch.tensor([[1533, 1534, 1535]] * 2, dtype=torch.int32))
    if kind == "csa":
        assert tok["ki_tok"].shape == (2, 1536, w.d_I) and tok["ki_tok"].dtype == dt
        assert qry["qI"].shape == (2, 3, w.H_I, w.d_I) and qry["qI"].dtype == dt
        assert qry["w_idx"].shape == (2, 3, w.H_I) and qry["w_idx"].dtype == torch.float32
    else:
        assert "ki_tok" not in tok and "qI" not in qry and "w_idx" not in qry


def test_bf16_is_the_rounded_f32_draw():
    w32 = small("csa", L=1024)
    tok32, tok16 = synth.make_tokens(w32, "cpu"), synth.make_tokens(w32.scaled(dtype="bf16"), "cpu")
    for name in ("k_tok", "v_tok", "ki_tok"):
        assert torch.equal(tok32[name].to(torch.bfloat16), tok16[name]), name
    assert torch.equal(tok32["gate"], tok16["gate"])


def test_scales_of_the_draws():
    w = small("csa", B=2, L=4096)
    tok, qry = synth.make_tokens(w, "cpu"), synth.make_queries(w, "cpu")
    for name, width in (("k_tok", w.d), ("v_tok", w.d), ("ki_tok", w.d_I)):
        x = tok[name].double()
        assert abs(x.mean().item()) < 0.02 / math.sqrt(width), name
        assert abs(x.std().item() * math.sqrt(width) - 1) < 0.02, name
    assert abs(tok["gate"].double().std().item() - 1) < 0.03
    wi = qry["w_idx"]
    assert (wi >= 0).all() and (wi < 1).all()


def test_different_sequences_are_different_draws():
    tok = synth.make_tokens(small("csa", B=2, L=1024), "cpu")
    assert not torch.equal(tok["k_tok"][0], tok["k_tok"][1])
    assert not torch.equal(tok["gate"][0], tok["gate"][1])


def test_rope_rotates_each_interleaved_pair_by_position_times_frequency():
    w0 = small("csa", L=1024, d=64, rope_dims=16)
    plain = synth.make_tokens(w0.scaled(rope_dims=0), "cpu")["k_tok"][0].double()
    rot = synth.make_tokens(w0, "cpu")["k_tok"][0].double()
    # dims past the rotary ones are untouched, position 0 is not rotated
    assert torch.equal(plain[:, 16:], rot[:, 16:])
    assert torch.allclose(plain[0], rot[0], atol=1e-7)
    a, b = plain[:, 0:16:2], plain[:, 1:16:2]
    ra, rb = rot[:, 0:16:2], rot[:, 1:16:2]
    # a rotation keeps the length of every pair
    assert torch.allclose(a * a + b * b, ra * ra + rb * rb, rtol=1e-5, atol=1e-9)
    # the first pair has frequency 1: its angle is the position itself (mod 2 pi);
    # the last pair has frequency theta^(-14/16)
    pos = torch.arange(1024, dtype=torch.float64)
    for i, freq in ((0, 1.0), (7, 10000.0 ** (-14 / 16))):
        turn = torch.atan2(a[:, i] * rb[:, i] - b[:, i] * ra[:, i],
                           a[:, i] * ra[:, i] + b[:, i] * rb[:, i])
        want = torch.remainder(pos * freq + math.pi, 2 * math.pi) - math.pi
        err = torch.remainder(turn - want + math.pi, 2 * math.pi) - math.pi
        assert err.abs().max() < 1e-4, i


def test_query_rope_uses_the_query_positions():
    w = small("csa", L=1024, d=64, rope_dims=16, Tq=4)
    q = synth.make_queries(w, "cpu")["q"][0].double()              # [Tq, H, d]
    q0 = synth.make_queries(w.scaled(rope_dims=0), "cpu")["q"][0].double()
    pos = torch.arange(1020, 1024, dtype=torch.float64)
    turn = torch.atan2(q0[..., 0] * q[..., 1] - q0[..., 1] * q[..., 0],
                       q0[..., 0] * q[..., 0] + q0[..., 1] * q[..., 1])
    want = torch.remainder(pos + math.pi, 2 * math.pi) - math.pi
    err = torch.remainder(turn - want[:, None] + math.pi, 2 * math.pi) - math.pi
    assert err.abs().max() < 1e-4


def test_plant_blocks_adds_the_stated_component_to_the_chosen_blocks_only():
    w = small("csa", B=2, L=8192, plant_frac=0.01, plant_sigma=3.0)
    tok, qry = synth.make_tokens(w, "cpu"), synth.make_queries(w, "cpu")
    before = tok["ki_tok"].clone()
    n_elig = 1900
    blocks = synth.plant_blocks(w, tok, qry, n_elig)
    n_plant = round(0.01 * w.n_blocks)
    assert blocks.shape == (2, n_plant)
    amp = 3.0 / math.sqrt(w.d_I)
    for b in range(2):
        bl = blocks[b]
        assert (bl[1:] > bl[:-1]).all() and bl.min() >= 0 and bl.max() < n_elig
        u = (qry["w_idx"][b, -1, :, None].double() * qry["qI"][b, -1].double()).sum(0)
        u_hat = u / u.norm()
        delta = (tok["ki_tok"][b] - before[b]).double()            # [L, d_I]
        planted = torch.zeros(w.L, dtype=torch.bool)
        for j in bl.tolist():
            planted[j * w.m:(j + 1) * w.m] = True
        assert (delta[~planted] == 0).all()
        d = delta[planted]
        assert torch.allclose(d, amp * u_hat.expand_as(d), atol=1e-6)
        # the projection of each planted key on u_hat grows by plant_sigma standard
        # deviations of a key's projection (1/sqrt(d_I))
        proj = d @ u_hat
        assert torch.allclose(proj, torch.full_like(proj, amp), rtol=1e-5)
    # the same seed plants the same blocks
    tok2 = synth.make_tokens(w, "cpu")
    assert torch.equal(synth.plant_blocks(w, tok2, qry, n_elig), blocks)
    assert torch.equal(tok2["ki_tok"], tok["ki_tok"])


@pytest.mark.parametrize("pad_frac", [0.0, 0.25])
def test_random_index_sets_are_distinct_ascending_and_padded(pad_frac):
    n_valid = torch.tensor([[0, 5, 40], [64, 3, 1000]], dtype=torch.int32)
    idx = synth.random_index_sets(2, 3, 16, n_valid, "cpu", seed=7, pad_frac=pad_frac)
    assert idx.shape == (2, 3, 16) and idx.dtype == torch.int32
    for b in range(2):
        for t in range(3):
            n = int(n_valid[b, t])
            take = min(16, n)
            take -= int(round(pad_frac * take))
            row = idx[b, t].tolist()
            sel = [v for v in row if v >= 0]
            assert row[len(sel):] == [-1] * (16 - len(sel))
            assert len(sel) == max(take, 0)
            assert sel == sorted(set(sel)) and all(0 <= v < n for v in sel)
    again = synth.random_index_sets(2, 3, 16, n_valid, "cpu", seed=7, pad_frac=pad_frac)
    assert torch.equal(idx, again)


def test_workloads_are_consistent():
    for name, w in synth.WORKLOADS.items():
        assert w.name == name and w.kind in ("csa", "hca")
        assert w.L % w.m == 0 and w.Tq <= w.L
        assert w.rope_dims % 2 == 0 and w.rope_dims <= w.d
        if w.kind == "hca":
            assert w.m == 128
        else:
            assert w.m == 4 and w.k > 0
        assert w.n_win == 128
    assert np.isclose(synth.WORKLOADS["csa_decode_1m"].plant_frac, 0.01)

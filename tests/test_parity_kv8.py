"""Compressed K/V in the FP8 format (HA_FMT_KV8; "DeepSeek-V4 深度研究剖析" §8: the KV
cache keeps its RoPE dims in BF16 and the other dims in FP8) against the oracle's
format of reading c23 (fp8_kv_encode / fp8_kv_decode / fp8_kv_pack).

  * compressor (m = 4 and m = 128 kernels): every sampled entry's 608-byte row
    decodes to the oracle's encoding of its float64 compressed row, except where a
    quantization decision sits near a rounding midpoint: the kernel decides on its
    float32 sum of m gated rows, the oracle on the float64 one, and the two differ
    by at most about m * 2^-24 relative (float32 accumulation of m terms whose
    weights sum to 1), so scales may differ by 2 m 2^-24 relative and codes where
    x / scale lies within max(1e-5, 2 m 2^-24) of a midpoint;
  * attention (decode over a selection with padding, ineligible and out-of-range
    entries in any order; HCA decode; prefill; the fused steps): against the
    oracle's attention over the decoded rows of the GPU's own cache; the kernels
    widen code * scale to bfloat16 before the tensor cores, which the bfloat16
    tolerance covers.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B
from long_context_hybrid_02_b300 import synth
from long_context_hybrid_02_b300.pipeline import HybridLayer, params_for
from tests._harness import assert_close, assert_lse_close, assert_topk_match, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _decoded(rows_u8):
    """[n, 608] uint8 rows -> [n, 512] float64 values they stand for."""
    return np.stack([O.fp8_kv_decode(*O.fp8_kv_unpack(r)) for r in rows_u8])


def _near_midpoint(v, lo, hi, rel=1e-5):
    return abs(v - 0.5 * (lo + hi)) <= rel * max(abs(v), 1e-30)


def _check_rows(w, tok, layer, b, blocks, names):
    for name, cname in names:
        rows = getattr(layer, cname)[b].cpu().numpy()
        for j in blocks:
            blk = slice(j * w.m, (j + 1) * w.m)
            x = O.compress(np64(tok[name][b, blk]), np64(tok["gate"][b, blk]), w.m, 0, 1)[0]
            rope_o, codes_o, scale_o = O.fp8_kv_encode(x)
            rope_g, codes_g, scale_g = O.fp8_kv_unpack(rows[j])
            assert_close(rope_g, rope_o, "bf16", f"{cname}[{b},{j}] rope")
            x32 = x[64:].reshape(7, 64).astype(np.float32)
            acc = 2.0 * w.m * 2.0 ** -24                  # float32 sum of m terms vs float64
            for g in range(7):
                assert abs(scale_g[g] - scale_o[g]) <= acc * scale_o[g], (cname, b, j, g)
                s = np.float32(scale_o[g])
                for e in np.nonzero(codes_g[g] != codes_o[g])[0]:
                    q = float(np.float32(x32[g, e]) / s)
                    assert _near_midpoint(abs(q), abs(codes_g[g, e]), abs(codes_o[g, e]),
                                          rel=max(1e-5, acc)), (cname, b, j, g, e)


@pytest.mark.parametrize("name", ["csa_decode_64k_kv8", "hca_decode_128k_kv8"])
def test_compressor_writes_fp8_rows(name):
    w = synth.WORKLOADS[name].scaled(B=2, L=16384)
    tok = synth.make_tokens(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache()
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    for b in range(w.B):
        blocks = list(rng.integers(0, w.n_blocks, 16)) + [0, w.n_blocks - 1]
        _check_rows(w, tok, layer, b, blocks, (("k_tok", "ck"), ("v_tok", "cv")))


def test_kv8_decode_over_messy_selections():
    """Given index sets (unsorted, -1, ineligible, beyond n_cap, some rows empty)
    over FP8 rows: the widening packs the valid entries first."""
    w = synth.WORKLOADS["csa_decode_64k_kv8"].scaled(B=5, L=8192)
    tok = synth.make_tokens(w, DEV)
    qry = synth.make_queries(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache()
    ctx = [8192, 8000, 129, 700, 140]
    ne = [O.n_eligible(c - 1, w.n_win, w.m) for c in ctx]
    idx = synth.random_index_sets(w.B, 1, w.k, torch.tensor(ne).reshape(w.B, 1), "cpu", 4)[:, 0].clone()
    idx[0] = idx[0][torch.randperm(w.k, generator=torch.Generator().manual_seed(2))]
    idx[0, 5], idx[0, 6], idx[0, 7] = -1, ne[0] + 2, 10 ** 6
    idx[1, 100:] = -1
    ctx_t = torch.tensor(ctx, dtype=torch.int32, device=DEV)
    o = torch.empty((w.B, w.H, w.d), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device=DEV)
    B.ha_device_error(clear=True)
    B.hybrid_attn_decode(layer.p, qry["q"][:, 0].contiguous(), layer.ck, layer.cv, layer.n_cap,
                         idx.to(DEV), tok["k_tok"], tok["v_tok"], w.L, ctx_t, o, lse,
                         (layer.ws.data_ptr(), layer.ws.numel()))
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    CK, CV = layer.ck.cpu().numpy(), layer.cv.cpu().numpy()
    for b, c in enumerate(ctx):
        t = c - 1
        lo = max(0, t - w.n_win + 1)
        ro, rl = O.prefill_query(np64(qry["q"][b, 0]), idx[b].numpy(), _decoded(CK[b]),
                                 _decoded(CV[b]), np64(tok["k_tok"][b, lo:c]),
                                 np64(tok["v_tok"][b, lo:c]), t, n_win=w.n_win, m=w.m,
                                 scale=1 / math.sqrt(w.d), tok_base=lo)
        assert_close(np64(o[b]), ro, "bf16", f"o[{b}]")
        assert_lse_close(np64(lse[b]), rl, "bf16", f"lse[{b}]")


@pytest.mark.parametrize("name", ["csa_decode_64k_kv8", "hca_decode_128k_kv8"])
def test_kv8_fused_step(name):
    w = synth.WORKLOADS[name].scaled(B=3, L=16384)
    tok = synth.make_tokens(w, DEV)
    qry = synth.make_queries(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache(n_blk=w.n_blocks - 1)
    ctx = torch.tensor([w.L, w.L - 1, w.L - 200], dtype=torch.int32, device=DEV)
    B.ha_device_error(clear=True)
    layer.decode_step_fused(qry["q"][:, 0].contiguous(), ctx, qry.get("qI"), qry.get("w_idx"))
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    CK, CV = layer.ck.cpu().numpy(), layer.cv.cpu().numpy()
    for b in range(w.B):
        c = int(ctx[b])
        t = c - 1
        ne = O.n_eligible(t, w.n_win, w.m)
        gi = None
        if w.kind == "csa":
            ref_scores = O.index_scores(np64(qry["qI"][b, 0]), np64(qry["w_idx"][b, 0]),
                                        np64(layer.cki[b, :ne]))
            gi = layer.idx[b, 0].cpu().numpy()
            assert_topk_match(gi, O.topk_select(ref_scores, w.k), ref_scores, w.k, f"top-k[{b}]")
        lo = t - w.n_win + 1
        ro, rl = O.prefill_query(np64(qry["q"][b, 0]), gi, _decoded(CK[b, :ne]), _decoded(CV[b, :ne]),
                                 np64(tok["k_tok"][b, lo:c]), np64(tok["v_tok"][b, lo:c]), t,
                                 n_win=w.n_win, m=w.m, scale=1 / math.sqrt(w.d), tok_base=lo)
        assert_close(np64(layer.o[b, 0]), ro, "bf16", f"o[{b}]")
        assert_lse_close(np64(layer.lse[b, 0]), rl, "bf16", f"lse[{b}]")


def test_kv8_prefill_rows():
    w = synth.WORKLOADS["csa_decode_64k_kv8"].scaled(B=1, L=4096, Tq=16)
    tok = synth.make_tokens(w, DEV)
    qry = synth.make_queries(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache()
    B.ha_device_error(clear=True)
    layer.prefill_chunk(qry["q"], qry["q_pos"], qry["qI"], qry["w_idx"])
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    CK, CV = _decoded(layer.ck[0].cpu().numpy()), _decoded(layer.cv[0].cpu().numpy())
    K, V = np64(tok["k_tok"][0]), np64(tok["v_tok"][0])
    for i in range(w.Tq):
        t = int(qry["q_pos"][0, i])
        ro, rl = O.prefill_query(np64(qry["q"][0, i]), layer.idx[0, i].cpu().numpy(), CK, CV, K, V,
                                 t, n_win=w.n_win, m=w.m, scale=1 / math.sqrt(w.d))
        assert_close(np64(layer.o[0, i]), ro, "bf16", f"o[{i}]")
        assert_lse_close(np64(layer.lse[0, i]), rl, "bf16", f"lse[{i}]")

"""The FP4 indexer with bfloat16 index scores (HA_FMT_IDX4; "DeepSeek-V4 深度研究剖析"
§8: the Lightning Indexer computes in FP4, its scores are kept in BF16) against the
oracle's format of reading c24 (fp4_encode / fp4_decode / fp4_pack).

  * compressor: every sampled block's 80-byte FP4 key row decodes to the oracle's
    encoding of its float64 compressed row, except where the quantization decision
    sits within 1e-5 (relative) of a rounding midpoint: the kernel decides on its
    float32 sum, the oracle on the float64 one;
  * indexer: scores of the GPU's own FP4 key rows and of the query quantized inside
    the kernel (the oracle quantizes the same bfloat16 query with the same float32
    decisions) equal the oracle's float64 scores rounded to bfloat16, up to one
    bfloat16 unit where the float32 sum lands across a rounding midpoint;
  * top-k on those bfloat16 scores is exact (ties by the smaller index);
  * the fused decode step through the FP4 indexer: selection exact on its own
    scores, attention against the oracle over that selection.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B
from long_context_hybrid_02_b300 import synth
from long_context_hybrid_02_b300.pipeline import HybridLayer
from tests._harness import assert_close, assert_lse_close, assert_sorted_unique, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"
GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


@pytest.fixture(scope="module")
def fp4():
    w = synth.WORKLOADS["csa_decode_64k_fp4"].scaled(B=4, L=16384)
    tok = synth.make_tokens(w, DEV)
    qry = synth.make_queries(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache()
    torch.cuda.synchronize()
    yield w, tok, qry, layer
    del layer, tok
    torch.cuda.empty_cache()


def _near_midpoint(v, lo, hi, rel=1e-5):
    mid = 0.5 * (lo + hi)
    return abs(v - mid) <= rel * max(abs(v), 1e-30)


def test_compressor_writes_the_fp4_rows_of_the_compressed_keys(fp4):
    w, tok, qry, layer = fp4
    rng = np.random.default_rng(5)
    rows = layer.cki.cpu().numpy()
    mismatched = checked = 0
    for b in range(w.B):
        for j in list(rng.integers(0, w.n_blocks, 40)) + [0, w.n_blocks - 1]:
            blk = slice(j * w.m, (j + 1) * w.m)
            x = O.compress(np64(tok["ki_tok"][b, blk]), np64(tok["gate"][b, blk]), w.m, 0, 1)  # float64
            codes_o, scale_o = O.fp4_encode(x)
            codes_g, scale_g = O.fp4_unpack(rows[b, j][None])
            assert (rows[b, j, 72:] == rows[b, j, 72:]).all()
            x32 = x.reshape(8, 16).astype(np.float32)
            for g in range(8):
                checked += 16
                if scale_g[0, g] != scale_o[0, g]:
                    # the scale decision: amax / 6 within 1e-5 of the midpoint of the two
                    amax = float(np.abs(x32[g]).max()) / 6.0
                    assert _near_midpoint(amax, scale_g[0, g], scale_o[0, g]), (b, j, g)
                    mismatched += 16
                    continue
                s = scale_o[0, g]
                for e in np.nonzero(codes_g[0, g] != codes_o[0, g])[0]:
                    q = float(x32[g, e]) / s
                    assert _near_midpoint(abs(q), abs(codes_g[0, g, e]), abs(codes_o[0, g, e])), (b, j, g, e)
                    mismatched += 1
    assert mismatched <= checked * 1e-3, (mismatched, checked)


def test_fp4_scores_and_exact_topk_on_them(fp4):
    w, tok, qry, layer = fp4
    qp = qry["q_pos"]
    B.csa_index_scores(layer.p, qry["qI"], qry["w_idx"], layer.cki, layer.n_cap, qp, 1, layer.scores)
    B.csa_topk(layer.p, layer.scores, layer.n_cap, qp, 1, layer.idx, (layer.ws.data_ptr(), layer.ws.numel()))
    torch.cuda.synchronize()
    t = w.L - 1
    ne = O.n_eligible(t, w.n_win, w.m)
    rows = layer.cki.cpu().numpy()
    exact = total = 0
    for b in range(w.B):
        keys = O.fp4_decode(*O.fp4_unpack(rows[b, :ne]))                   # what the kernel read
        q4 = O.fp4_decode(*O.fp4_encode(np64(qry["qI"][b, 0])))            # the kernel's rule
        ref = O.round_to_bf16(O.index_scores(q4, np64(qry["w_idx"][b, 0]), keys))
        got = np64(layer.scores[b, 0, :ne])
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
        assert (np.abs(got - ref) <= ulp).all(), b
        exact += int((got == ref).sum())
        total += ne
        gi = layer.idx[b, 0].cpu().numpy()
        assert_sorted_unique(gi, ne, w.k, f"idx[{b}]")
        assert gi.tolist() == O.topk_select(got, w.k).tolist(), b    # exact on the same scores
    assert exact >= 0.99 * total, (exact, total)


def test_fp4_decode_step_end_to_end(fp4):
    w, tok, qry, layer = fp4
    ctx = torch.tensor([w.L, w.L - 1, w.L - 4, w.L - 77], dtype=torch.int32, device=DEV)
    B.ha_device_error(clear=True)
    layer.decode_step_fused(qry["q"][:, 0].contiguous(), ctx, qry["qI"], qry["w_idx"])
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    rows = layer.cki.cpu().numpy()
    for b in range(w.B):
        c = int(ctx[b])
        t = c - 1
        ne = O.n_eligible(t, w.n_win, w.m)
        got = np64(layer.scores[b, 0, :ne])
        gi = layer.idx[b, 0].cpu().numpy()
        assert gi.tolist() == O.topk_select(got, w.k).tolist(), b
        keys = O.fp4_decode(*O.fp4_unpack(rows[b, :ne]))
        q4 = O.fp4_decode(*O.fp4_encode(np64(qry["qI"][b, 0])))
        ref = O.round_to_bf16(O.index_scores(q4, np64(qry["w_idx"][b, 0]), keys))
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
        assert (np.abs(got - ref) <= ulp).all(), b
        lo = t - w.n_win + 1
        ro, rl = O.prefill_query(np64(qry["q"][b, 0]), gi, np64(layer.ck[b]), np64(layer.cv[b]),
                                 np64(tok["k_tok"][b, lo:c]), np64(tok["v_tok"][b, lo:c]), t,
                                 n_win=w.n_win, m=w.m, scale=1 / math.sqrt(w.d), tok_base=lo)
        assert_close(np64(layer.o[b, 0]), ro, "bf16", f"o[{b}]")
        assert_lse_close(np64(layer.lse[b, 0]), rl, "bf16", f"lse[{b}]")

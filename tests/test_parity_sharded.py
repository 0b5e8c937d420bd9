"""Context sharding of one long sequence (long_context_hybrid_02_b300.sharded) with
the library's kernels, on one GPU: the G shards run one after the other in one
process and the all-gathers are concatenations, so no kernel waits on another.
What this covers is what the kernels do for a shard: scoring and selecting over
the shard's own eligible range (shard_ctx_len), the global top k over the
gathered candidates, attention without the window on the shards that do not hold
the tail (k_tok = v_tok = NULL), and hybrid_attn_merge.  The collectives and the
exchange on several processes are covered on the CPU (test_multi_rank_cpu.py).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B
from long_context_hybrid_02_b300 import sharded as S
from long_context_hybrid_02_b300 import synth
from long_context_hybrid_02_b300.pipeline import HybridLayer, params_for
from tests._harness import assert_close, assert_lse_close, assert_topk_match, np64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _emulate(shards, q, qI, w_idx, t, ops):
    cands = [ops.candidates(sh, qI, w_idx, t) for sh in shards]
    all_s = torch.cat([c[0] for c in cands])
    all_i = torch.cat([c[1] for c in cands])
    sel = ops.select(shards[0].p, all_s, all_i)
    parts = [ops.partial(sh, q, sel, t) for sh in shards]
    o, lse = ops.merge(shards[0].p, torch.stack([p[0] for p in parts]),
                       torch.stack([p[1] for p in parts]), q.dtype)
    return o, lse, sel


@pytest.mark.parametrize("name,G,ctx", [("csa_decode_64k", 4, 65536), ("csa_decode_64k", 3, 60001),
                                        ("tiny_csa", 2, 1024), ("tiny_csa", 5, 700)])
def test_sharded_decode_matches_the_oracle(name, G, ctx):
    w = synth.WORKLOADS[name].scaled(B=1)
    if name == "csa_decode_64k":
        w = w.scaled(L=65536)
    tok = synth.make_tokens(w, DEV)
    qry = synth.make_queries(w, DEV)
    layer = HybridLayer(w, tok, DEV)
    layer.build_cache()                         # the whole sequence's compressed caches
    torch.cuda.synchronize()
    p = params_for(w)
    n = w.n_blocks
    shards = []
    for r in range(G):
        j0, j1 = S.shard_range(n, r, G)
        tail = r == G - 1
        shards.append(S.Shard(p=p, ck=layer.ck[:, j0:j1].contiguous(),
                              cv=layer.cv[:, j0:j1].contiguous(),
                              cki=layer.cki[:, j0:j1].contiguous(), j0=j0, j1=j1,
                              k_tok=tok["k_tok"] if tail else None,
                              v_tok=tok["v_tok"] if tail else None, tok_cap=w.L))
    t = ctx - 1
    q = qry["q"][0, 0].contiguous()
    B.ha_device_error(clear=True)
    o, lse, sel = _emulate(shards, q, qry["qI"][:, :1].contiguous(), qry["w_idx"][:, :1].contiguous(),
                           t, S.LibraryOps(DEV))
    torch.cuda.synchronize()
    assert B.ha_device_error() == 0
    ne = O.n_eligible(t, w.n_win, w.m)
    ref_scores = O.index_scores(np64(qry["qI"][0, 0]), np64(qry["w_idx"][0, 0]),
                                np64(layer.cki[0, :ne]))
    gi = sel.cpu().numpy()
    assert_topk_match(gi, O.topk_select(ref_scores, w.k), ref_scores, w.k, "global top-k")
    CK, CV = np64(layer.ck[0]), np64(layer.cv[0])
    lo = max(0, t - w.n_win + 1)
    ro, rl = O.prefill_query(np64(q), gi, CK, CV, np64(tok["k_tok"][0, lo:ctx]),
                             np64(tok["v_tok"][0, lo:ctx]), t, n_win=w.n_win, m=w.m,
                             scale=1 / math.sqrt(w.d), tok_base=lo)
    assert_close(np64(o), ro, w.dtype, "o")
    assert_lse_close(np64(lse), rl, w.dtype, "lse")


@pytest.mark.parametrize("rows,S_,H,d,dt", [(3, 5, 64, 512, "f32"), (2, 3, 64, 512, "bf16"),
                                             (2, 1700, 10, 136, "bf16"), (1, 37, 9, 1024, "f32")])
def test_merge_call_against_the_oracle_merge(rows, S_, H, d, dt):
    """hybrid_attn_merge on random partials (some without keys) against the oracle's
    merge_partials: head counts that do not fill a CTA's heads, head dims that do
    not fill a 512-dim pass, split counts past one group of four and past the
    default shared-memory limit (1,700 splits)."""
    g = torch.Generator(device=DEV).manual_seed(3)
    o_part = torch.randn((rows, S_, H, d), generator=g, device=DEV)
    lse_part = torch.randn((rows, S_, H), generator=g, device=DEV) * 4
    last = min(rows - 1, 2)
    lse_part[min(rows - 1, 1), 2] = float("-inf")    # a split without keys
    lse_part[last, :, 5] = float("-inf")             # a head with no key in any part
    p = B.make_params(rows, H, d, 128, 4, dtype=B.F32 if dt == "f32" else B.BF16)
    o = torch.empty((rows, H, d), device=DEV, dtype=torch.float32 if dt == "f32" else torch.bfloat16)
    lse = torch.empty((rows, H), device=DEV)
    B.hybrid_attn_merge(p, rows, S_, o_part, lse_part, o, lse)
    torch.cuda.synchronize()
    for r in range(rows):
        ro, rl = O.merge_partials(np64(o_part[r]), np64(lse_part[r]))
        assert_close(np64(o[r]), ro, dt, f"o[{r}]")
        assert_lse_close(np64(lse[r]), rl, "f32", f"lse[{r}]")
    assert (np64(o[last, 5]) == 0).all() and np.isneginf(np64(lse[last, 5]))

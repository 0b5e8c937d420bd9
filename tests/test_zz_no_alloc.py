"""hybrid_attn_decode_static: decode attention for callers that cannot allocate.

Engine plugins that only receive a layer's input/output pointers, code that
lives inside another runtime's memory pool, and serving loops that must not
call cudaMalloc (it synchronises the device) cannot pass a workspace.  This
entry point keeps the split-KV partials in the library's own fixed 32 MiB device
array instead.  These tests check that it gives the same outputs as
hybrid_attn_decode with a caller-allocated workspace, on two calls in a row
(the second call must not see stale partials of the first), and that a problem
too large for the fixed array is refused before anything runs.

This file is collected last on purpose, so that a run stopping at the first
failure has already run every other test.
"""
import math
import os

import pytest
import torch

from long_context_hybrid_02_b300 import binding as B
from long_context_hybrid_02_b300 import synth
from tests._harness import assert_close, assert_lse_close, np64

A = 1 << 20      # aligned fake address: the refusal happens before any CUDA call


def test_static_decode_refuses_problems_beyond_the_fixed_scratch():
    if not os.path.exists(B.LIB_PATH):
        pytest.skip("the CUDA library is not built")
    B.load_library()
    # float32 storage (the CUDA-core path splits every 128 keys): 64 sequences x 128
    # heads x 512 dims over 8,192 + 128 keys needs ~1 GB of partials
    p = B.make_params(64, 128, 512, 128, 128, dtype=B.F32)
    need = B.ha_workspace_size(p, B.OP_DECODE, 1, 8192, False)
    assert need > B.STATIC_SCRATCH_BYTES
    with pytest.raises(B.HAError) as e:
        B.hybrid_attn_decode_static(p, A, A, A, 8192, None, A, A, 1 << 17, A, A, None, stream=0)
    assert e.value.code == 4 and "static scratch" in str(e.value)


def _problem(kind, dtype, B_, L, H, d, k, seed):
    w = synth.Workload(f"static_{kind}", kind, B_, L, H, d, 128, 4 if kind == "csa" else 128, k,
                       1, 8, dtype, seed=seed)
    dev = "cuda"
    tok = synth.make_tokens(w, dev)
    qry = synth.make_queries(w, dev)
    n_cap = w.n_blocks
    dt = w.torch_dtype
    ck = synth.gaussian((w.B, n_cap, d), dev, seed + 1, 1 / math.sqrt(d), dt)
    cv = synth.gaussian((w.B, n_cap, d), dev, seed + 2, 1 / math.sqrt(d), dt)
    ne = max(0, L - 128) // w.m
    idx = None
    if kind == "csa":
        idx = synth.random_index_sets(w.B, 1, k, torch.full((w.B, 1), ne), dev, seed)[:, 0].contiguous()
    p = B.make_params(w.B, H, d, 128, w.m, k, 1, 8, B.F32 if dtype == "f32" else B.BF16)
    return w, p, tok, qry, ck, cv, idx, n_cap


def _run_both(w, p, tok, q, ck, cv, idx, n_cap, ctx_len):
    dt = w.torch_dtype
    o_ref = torch.empty((w.B, w.H, w.d), dtype=dt, device="cuda")
    lse_ref = torch.empty((w.B, w.H), dtype=torch.float32, device="cuda")
    ws = torch.empty(B.ha_workspace_size(p, B.OP_DECODE, 1, n_cap, idx is not None),
                     dtype=torch.uint8, device="cuda")
    B.hybrid_attn_decode(p, q, ck, cv, n_cap, idx, tok["k_tok"], tok["v_tok"], w.L, ctx_len,
                         o_ref, lse_ref, ws)
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    B.hybrid_attn_decode_static(p, q, ck, cv, n_cap, idx, tok["k_tok"], tok["v_tok"], w.L,
                                ctx_len, o, lse)
    torch.cuda.synchronize()
    return o_ref, lse_ref, o, lse


@pytest.mark.gpu
@pytest.mark.parametrize("kind,dtype,B_,L,H,d,k,uses_scratch", [
    # tensor cores: few rows, so every row's keys are cut into splits whose float32
    # partials go through the scratch (8 rows of 512 + 128 keys, 4 rows of 511 + 128,
    # one row of 2,047 + 128)
    ("csa", "bf16", 8, 16384, 64, 512, 512, True),
    ("hca", "bf16", 4, 65536, 64, 512, 1, True),
    ("hca", "bf16", 1, 262144, 64, 512, 1, True),
    # tensor cores, 160 rows: one split per row, written directly (no scratch)
    ("hca", "bf16", 160, 4096, 64, 512, 1, False),
    # CUDA cores: split partials of every row go through the scratch
    ("csa", "f32", 2, 1024, 8, 64, 16, True),
])
def test_static_decode_matches_workspace_decode_twice_in_a_row(kind, dtype, B_, L, H, d, k,
                                                              uses_scratch):
    w, p, tok, qry, ck, cv, idx, n_cap = _problem(kind, dtype, B_, L, H, d, k, seed=40)
    need = B.ha_workspace_size(p, B.OP_DECODE, 1, n_cap, idx is not None)
    assert (need > 0) == uses_scratch, need
    assert need <= B.STATIC_SCRATCH_BYTES
    q1 = qry["q"][:, 0].contiguous()
    ctx1 = qry["ctx_len"]
    # first call
    o_ref, lse_ref, o, lse = _run_both(w, p, tok, q1, ck, cv, idx, n_cap, ctx1)
    assert_close(np64(o), np64(o_ref), dtype, "o (first call)")
    assert_lse_close(np64(lse), np64(lse_ref), dtype, "lse (first call)")
    # second call with other queries and shorter contexts: the scratch still
    # holds the first call's partials, which must not leak into the result
    q2 = synth.gaussian(q1.shape, "cuda", 99, 1 / math.sqrt(d), q1.dtype)
    ctx2 = (ctx1 - torch.arange(w.B, device="cuda", dtype=torch.int32) * 37).contiguous()
    o_ref2, lse_ref2, o2, lse2 = _run_both(w, p, tok, q2, ck, cv, idx, n_cap, ctx2)
    assert_close(np64(o2), np64(o_ref2), dtype, "o (second call)")
    assert_lse_close(np64(lse2), np64(lse_ref2), dtype, "lse (second call)")
    assert not torch.equal(o2, o)

"""One hybrid-attention layer driven through the C ABI.

`HybridLayer` owns the device buffers of one layer (compressed caches, scores,
selected indices, outputs, workspace) and issues the library calls of a decode
step or a prefill chunk in the order the method runs them: compress the block
that just completed -> score every eligible entry -> select the top k -> attend
to the selection plus the window (CSA); compress -> attend to every eligible
entry plus the window (HCA).  `decode_step_fused` issues the same stages through
one call (csa_decode_step / hca_decode_step).  With a `CacheState` the layer also
takes ragged appends of new tokens into ring-buffered per-token caches and
compresses the blocks they complete.  Torch only allocates memory, copies the
caller's new token rows into their cache slots and provides the stream; every
stage of the method runs in the library's CUDA kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from .cache_state import CacheState
from .synth import Workload


def params_for(w: Workload, Tq_override: int | None = None) -> B.Params:
    return B.make_params(w.B, w.H, w.d, w.n_win, w.m, w.k if w.kind == "csa" else 1,
                         w.H_I if w.kind == "csa" else 1, w.d_I if w.kind == "csa" else 8,
                         B.F32 if w.dtype == "f32" else B.BF16, B.ELIG_DISJOINT, 0.0, w.fmt)


class HybridLayer:
    def __init__(self, w: Workload, tokens: dict, device="cuda", n_cap: int | None = None,
                 tok_cap: int | None = None, state: CacheState | None = None):
        self.w = w
        self.device = device
        self.p = params_for(w)
        self.csa = w.kind == "csa"
        self.tok = tokens
        self.tok_cap = tok_cap or tokens["k_tok"].shape[1]
        self.n_cap = n_cap or w.n_blocks
        dt = w.torch_dtype
        self.kv8 = bool(w.fmt & B.FMT_KV8)
        if self.kv8:                        # 608-byte FP8 rows of the compressed K / V
            self.ck = torch.empty((w.B, self.n_cap, B.KV8_ROW_BYTES), dtype=torch.uint8, device=device)
            self.cv = torch.empty((w.B, self.n_cap, B.KV8_ROW_BYTES), dtype=torch.uint8, device=device)
        else:
            self.ck = torch.empty((w.B, self.n_cap, w.d), dtype=dt, device=device)
            self.cv = torch.empty((w.B, self.n_cap, w.d), dtype=dt, device=device)
        self.fp4 = bool(w.fmt & B.FMT_IDX4)
        if not self.csa:
            self.cki = None
        elif self.fp4:                      # 80-byte FP4 rows of the indexer keys
            self.cki = torch.empty((w.B, self.n_cap, B.IDX4_ROW_BYTES), dtype=torch.uint8,
                                   device=device)
        else:
            self.cki = torch.empty((w.B, self.n_cap, w.d_I), dtype=dt, device=device)
        Tq = w.Tq
        sdt = torch.bfloat16 if self.fp4 else torch.float32
        self.scores = torch.empty((w.B, Tq, self.n_cap), dtype=sdt, device=device) if self.csa else None
        self.idx = torch.empty((w.B, Tq, w.k), dtype=torch.int32, device=device) if self.csa else None
        self.o = torch.empty((w.B, Tq, w.H, w.d), dtype=dt, device=device)
        self.lse = torch.empty((w.B, Tq, w.H), dtype=torch.float32, device=device)
        op = B.OP_DECODE if w.decode else B.OP_PREFILL
        nb = B.ha_workspace_size(self.p, op, Tq, self.n_cap, self.csa)
        if self.csa:
            nb = max(nb, B.ha_workspace_size(self.p, B.OP_TOPK, Tq, self.n_cap, True))
        if w.decode:
            nb = max(nb, B.ha_workspace_size(self.p, B.OP_DECODE_STEP, 1, self.n_cap, self.csa))
        self.state = state
        self.ws = torch.empty((max(nb, 16),), dtype=torch.uint8, device=device)
        self.blk_zero = torch.zeros((w.B,), dtype=torch.int32, device=device)
        # side stream for the decode step's compression (see decode_step)
        self._side = torch.cuda.Stream(device=device)
        self._fork = torch.cuda.Event()
        self._join = torch.cuda.Event()

    # ------------------------------------------------------------------ caches
    def compress(self, blk_begin: torch.Tensor, n_blk: int, stream=None):
        t = self.tok
        if self.csa:
            B.csa_compress_kv(self.p, t["k_tok"], t["v_tok"], t["ki_tok"], t["gate"], self.tok_cap,
                              blk_begin, n_blk, self.ck, self.cv, self.cki, self.n_cap, stream)
        else:
            B.hca_compress_kv(self.p, t["k_tok"], t["v_tok"], t["gate"], self.tok_cap, blk_begin,
                              n_blk, self.ck, self.cv, self.n_cap, stream)

    def build_cache(self, n_blk: int | None = None, stream=None):
        """Compress blocks 0 .. n_blk-1 of every sequence (all complete blocks by default)."""
        self.compress(self.blk_zero, self.n_cap if n_blk is None else n_blk, stream)

    # ------------------------------------------------------------------ steps
    def decode_step(self, q, ctx_len, new_blk, qI=None, w_idx=None, q_pos=None, stream=None):
        """One decode token per sequence.

        new_blk: int32 [B] index of the block completed by the newest token, or None
        when no block completed at this step.  q_pos = ctx_len - 1 (int32 [B, 1]).

        Under the disjoint eligibility rule a block is visible to a query only once it
        ends before the query's window.  The newest complete block ends at most m - 1
        tokens before the query, so with n_win >= m it is not visible to this step:
        its compression then runs on a side stream beside scoring, selection and
        attention, and the step's stream waits for it before returning.  Otherwise
        (overlap rule, or n_win < m) the block is compressed first.
        """
        main = torch.cuda.ExternalStream(B._stream(stream))
        joined = False
        if new_blk is not None:
            if self.p.elig == B.ELIG_DISJOINT and self.p.n_win >= self.p.m:
                self._fork.record(main)
                self._side.wait_event(self._fork)
                self.compress(new_blk, 1, self._side.cuda_stream)
                self._join.record(self._side)
                joined = True
            else:
                self.compress(new_blk, 1, stream)
        ws = (self.ws.data_ptr(), self.ws.numel())
        if self.csa:
            B.csa_index_scores(self.p, qI, w_idx, self.cki, self.n_cap, q_pos, 1, self.scores, stream)
            B.csa_topk(self.p, self.scores, self.n_cap, q_pos, 1, self.idx, ws, stream)
            B.hybrid_attn_decode(self.p, q, self.ck, self.cv, self.n_cap, self.idx,
                                 self.tok["k_tok"], self.tok["v_tok"], self.tok_cap, ctx_len,
                                 self.o, self.lse, ws, stream)
        else:
            B.hybrid_attn_decode(self.p, q, self.ck, self.cv, self.n_cap, None, self.tok["k_tok"],
                                 self.tok["v_tok"], self.tok_cap, ctx_len, self.o, self.lse, ws,
                                 stream)
        if joined:
            main.wait_event(self._join)
        return self.o

    def decode_step_fused(self, q, ctx_len, qI=None, w_idx=None, stream=None):
        """The decode step through one library call: the block completed by the
        newest token (if any) is compressed, then (CSA) scoring, selection and
        attention.  The newest token's rows must already be in the per-token caches."""
        t = self.tok
        ws = (self.ws.data_ptr(), self.ws.numel())
        if self.csa:
            B.csa_decode_step(self.p, q, qI, w_idx, t["k_tok"], t["v_tok"], t["ki_tok"], t["gate"],
                              self.tok_cap, ctx_len, self.ck, self.cv, self.cki, self.n_cap,
                              self.scores, self.idx, self.o, self.lse, ws, stream)
        else:
            B.hca_decode_step(self.p, q, t["k_tok"], t["v_tok"], t["gate"], self.tok_cap, ctx_len,
                              self.ck, self.cv, self.n_cap, self.o, self.lse, ws, stream)
        return self.o

    def append(self, rows: dict, n_new, stream=None):
        """Append n_new[b] tokens to sequence b ([V4-notes] §11.4: the tokens of an
        unfinished block stay in the per-token cache, the "tail", until their block
        completes).  rows[name]: [B, >= max(n_new), dim] device tensors of the new
        tokens' rows (k_tok, v_tok, gate and, for CSA, ki_tok); the first n_new[b]
        of sequence b are used.  They are copied to their ring slots, then the blocks
        they complete are compressed in one call.  Returns the new context lengths."""
        if self.state is None:
            raise RuntimeError("append needs a CacheState")
        n_new = np.asarray(n_new, dtype=np.int64).reshape(-1)
        slots = [self.state.slots(b, int(n_new[b])) for b in range(self.w.B)]
        blk_begin, n_blk = self.state.append(n_new)
        for name, dst in self.tok.items():
            for b in range(self.w.B):
                if n_new[b] == 0:
                    continue
                idx = torch.as_tensor(slots[b], device=dst.device)
                dst[b].index_copy_(0, idx, rows[name][b, :int(n_new[b])].to(dst.dtype))
        if n_blk > 0:
            self.compress(torch.as_tensor(blk_begin, device=self.device), n_blk, stream)
        return self.state.ctx.copy()

    def prefill_chunk(self, q, q_pos, qI=None, w_idx=None, stream=None):
        """Tq queries per sequence (their tokens and blocks already in the caches)."""
        Tq = q.shape[1]
        ws = (self.ws.data_ptr(), self.ws.numel())
        if self.csa:
            B.csa_index_scores(self.p, qI, w_idx, self.cki, self.n_cap, q_pos, Tq, self.scores, stream)
            B.csa_topk(self.p, self.scores, self.n_cap, q_pos, Tq, self.idx, ws, stream)
        B.hybrid_attn_prefill(self.p, q, q_pos, Tq, self.ck, self.cv, self.n_cap,
                              self.idx if self.csa else None, self.tok["k_tok"], self.tok["v_tok"],
                              self.tok_cap, self.o, self.lse, ws, stream)
        return self.o

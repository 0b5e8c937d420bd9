"""One long sequence's CSA layer spread over G GPUs (context sharding).

The compressed entries of the sequence ("DeepSeek-V4 深度研究剖析" §5.3: every m
tokens' KV and indexer key compressed into one entry) are cut into G contiguous
ranges, one per rank; the rank holding the last range also holds the per-token
rows of the sliding window (§5.2).  One decode query at position t then runs:

  1. every rank scores its eligible entries and keeps its local top k;
  2. the G x k candidates (score, global entry index) are all-gathered and the
     global top k taken from them.  This is the sequence's exact top k: an entry
     that k entries of the whole sequence do not beat is not beaten by k entries
     of its own range either, so it is among its rank's candidates.  Candidates
     are laid out rank by rank, each rank's in ascending index order, so their
     order is the global index order and the top-k's tie rule (smaller index
     first) is the global one;
  3. every rank attends to the selected entries of its range (the tail rank also
     to the window) and gets a partial (o_r, lse_r);
  4. the partials are all-gathered and merged: o = sum_r exp(lse_r - LSE) o_r
     (the one softmax over all keys, "EP 95 解读 DeepSeek-V4 论文" figure).

Every score, selection, attention and merge runs in the library's kernels; this
module only does the index bookkeeping of the exchange (plain torch indexing)
and the collectives (torch.distributed all-gather: NCCL between GPUs, any backend
in general).  The local compute goes through an `ops` object whose default is
`LibraryOps`; a multi-process test on the CPU can pass its own.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

from . import binding as B


def shard_range(n_entries: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced range [j0, j1) of compressed entries owned by `rank`."""
    return n_entries * rank // world, n_entries * (rank + 1) // world


def n_eligible(t: int, n_win: int, m: int, elig: int) -> int:
    """Entries visible to the query at position t (the library's eligibility rule)."""
    if t < 0:
        return 0
    return (t + 1) // m if elig == B.ELIG_OVERLAP else max(0, t + 1 - n_win) // m


def shard_ctx_len(t: int, j0: int, j1: int, n_win: int, m: int, elig: int) -> int:
    """Context length whose eligibility over a shard's own rows 0 .. j1-j0-1 is the
    global eligibility of entries j0 .. j1-1 for the query at position t."""
    n_loc = min(max(n_eligible(t, n_win, m, elig) - j0, 0), j1 - j0)
    return n_loc * m + (0 if elig == B.ELIG_OVERLAP else n_win)


def pack_candidates(scores: torch.Tensor, local_idx: torch.Tensor, j0: int):
    """A rank's local top k as candidates: float32 scores (-inf for padding) and
    int32 global entry indices (-1 for padding), in ascending index order."""
    valid = local_idx >= 0
    s = scores[local_idx.clamp(min=0).long()]
    s = torch.where(valid, s, torch.full_like(s, float("-inf")))
    g = torch.where(valid, local_idx + j0, torch.full_like(local_idx, -1))
    return s.contiguous(), g.to(torch.int32).contiguous()


def split_selection(global_idx: torch.Tensor, j0: int, j1: int) -> torch.Tensor:
    """The selected entries a rank owns, as its local indices (-1 elsewhere)."""
    mine = (global_idx >= j0) & (global_idx < j1)
    return torch.where(mine, global_idx - j0, torch.full_like(global_idx, -1)).to(torch.int32)


@dataclass
class Shard:
    """What one rank holds of the sequence: compressed rows j0 .. j1-1 (rows 0 ..
    j1-j0-1 of ck, cv, cki) and, on the tail rank, the per-token window caches."""
    p: B.Params                 # layer parameters with B = 1
    ck: torch.Tensor            # [1, j1 - j0, d]
    cv: torch.Tensor
    cki: torch.Tensor           # [1, j1 - j0, d_I]
    j0: int
    j1: int
    k_tok: torch.Tensor | None = None   # [1, tok_cap, d] on the tail rank only
    v_tok: torch.Tensor | None = None
    tok_cap: int = 0


class LibraryOps:
    """The local stages through the library (device tensors, current stream)."""

    def __init__(self, device):
        self.device = device

    def _i32(self, v):
        return torch.tensor([v], dtype=torch.int32, device=self.device)

    def candidates(self, sh: Shard, qI, w_idx, t):
        n_loc = sh.j1 - sh.j0
        ctx = shard_ctx_len(t, sh.j0, sh.j1, sh.p.n_win, sh.p.m, sh.p.elig)
        pos = self._i32(ctx - 1).reshape(1, 1)
        scores = torch.empty((1, 1, n_loc), dtype=torch.float32, device=self.device)
        idx = torch.empty((1, 1, sh.p.k), dtype=torch.int32, device=self.device)
        B.csa_index_scores(sh.p, qI, w_idx, sh.cki, n_loc, pos, 1, scores)
        ws = torch.empty(max(16, B.ha_workspace_size(sh.p, B.OP_TOPK, 1, n_loc, True)),
                         dtype=torch.uint8, device=self.device)
        B.csa_topk(sh.p, scores, n_loc, pos, 1, idx, ws)
        return pack_candidates(scores[0, 0], idx[0, 0], sh.j0)

    def select(self, p: B.Params, cand_scores, cand_idx):
        """Global top k of the gathered candidates (one row of G x k)."""
        n = cand_scores.numel()
        pg = B.make_params(1, p.H, p.d, p.n_win, p.m, p.k, p.H_I, p.d_I, p.dtype, B.ELIG_OVERLAP,
                           p.scale)
        pos = self._i32(n * p.m - 1).reshape(1, 1)           # overlap rule: all n eligible
        pick = torch.empty((1, 1, p.k), dtype=torch.int32, device=self.device)
        ws = torch.empty(max(16, B.ha_workspace_size(pg, B.OP_TOPK, 1, n, True)),
                         dtype=torch.uint8, device=self.device)
        B.csa_topk(pg, cand_scores.reshape(1, 1, n), n, pos, 1, pick, ws)
        pick = pick[0, 0]
        g = cand_idx[pick.clamp(min=0).long()]
        return torch.where(pick >= 0, g, torch.full_like(g, -1)).to(torch.int32)

    def partial(self, sh: Shard, q, global_sel, t):
        """Attention over the selected entries the shard owns (plus the window on the
        tail rank): (o_r float32 [H, d], lse_r [H])."""
        local = split_selection(global_sel, sh.j0, sh.j1).reshape(1, -1).contiguous()
        n_loc = sh.j1 - sh.j0
        if sh.k_tok is not None:                             # tail: real position, window
            ctx = self._i32(t + 1)
        else:
            ctx = self._i32(shard_ctx_len(t, sh.j0, sh.j1, sh.p.n_win, sh.p.m, sh.p.elig))
        o = torch.empty((1, sh.p.H, sh.p.d), dtype=q.dtype, device=self.device)
        lse = torch.empty((1, sh.p.H), dtype=torch.float32, device=self.device)
        ws = torch.empty(max(16, B.ha_workspace_size(sh.p, B.OP_DECODE, 1, n_loc, True)),
                         dtype=torch.uint8, device=self.device)
        B.hybrid_attn_decode(sh.p, q.reshape(1, sh.p.H, sh.p.d), sh.ck, sh.cv, n_loc, local,
                             sh.k_tok, sh.v_tok, sh.tok_cap, ctx, o, lse, ws)
        return o[0].float(), lse[0]

    def merge(self, p: B.Params, o_parts, lse_parts, out_dtype):
        G = o_parts.shape[0]
        o = torch.empty((1, p.H, p.d), dtype=out_dtype, device=self.device)
        lse = torch.empty((1, p.H), dtype=torch.float32, device=self.device)
        B.hybrid_attn_merge(p, 1, G, o_parts.reshape(1, G, p.H, p.d).contiguous(),
                            lse_parts.reshape(1, G, p.H).contiguous(), o, lse)
        return o[0], lse[0]


def _all_gather(x: torch.Tensor, world: int, group=None) -> torch.Tensor:
    """[world, *x.shape]: every rank's x, in rank order."""
    import torch.distributed as dist
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x.contiguous(), group=group)
    return torch.stack(parts)


def sharded_decode(sh: Shard, q, qI, w_idx, t: int, world: int, ops=None, group=None):
    """One decode query of a sharded sequence on this rank (every rank calls it with
    the same q, qI, w_idx and t); returns the merged (o [H, d], lse [H]) and the
    global selection (int32 [k], ascending, -1 padded), the same on every rank."""
    ops = ops or LibraryOps(q.device)
    cs, ci = ops.candidates(sh, qI, w_idx, t)
    all_s = _all_gather(cs, world, group).reshape(-1)
    all_i = _all_gather(ci, world, group).reshape(-1)
    sel = ops.select(sh.p, all_s, all_i)
    o_r, lse_r = ops.partial(sh, q, sel, t)
    o_all = _all_gather(o_r, world, group)
    lse_all = _all_gather(lse_r, world, group)
    o, lse = ops.merge(sh.p, o_all, lse_all, q.dtype)
    return o, lse, sel

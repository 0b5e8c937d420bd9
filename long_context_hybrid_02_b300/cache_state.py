"""Host-side bookkeeping of one layer's caches: which blocks to compress after an
append, and whether a ring of per-token slots is large enough.

The compressed caches hold one entry per complete block of m tokens; the tokens
of a block that is not complete yet stay only in the per-token buffer (the
"tail"), and the per-token buffer also serves the sliding window ("DeepSeek-V4
深度研究剖析" §11.4 lists these cache kinds: compressed KV, indexer KV, the SWA
state and the uncompressed tail).  The per-token buffer is `[B, tok_cap, ·]`
with token u of a sequence at slot u % tok_cap.

`CacheState.append(n_new)` records that sequence b received n_new[b] tokens (their
rows already written at `slots`) and returns the arguments of one compressor call
(`csa_compress_kv` / `hca_compress_kv`): per sequence the first block it completes
(-1 when it completes none) and one block count for the whole batch, the largest
number of blocks any sequence completed.  A sequence that completed fewer blocks
then also has some incomplete blocks compressed: harmless, because an entry is
eligible for a query only once its block is complete and lies before the window,
and the block is compressed again, from its complete rows, by the append that
completes it.  The ring check makes sure every token the step reads is still
resident: the window of the first new query and the first block completed.

Pure Python and numpy; it launches nothing.
"""
from __future__ import annotations

import numpy as np


class CacheState:
    def __init__(self, B: int, m: int, n_win: int, tok_cap: int, n_cap: int, ctx=None):
        if B < 1 or m < 1 or n_win < 1 or tok_cap < 1 or n_cap < 1:
            raise ValueError("B, m, n_win, tok_cap and n_cap must be positive")
        self.B, self.m, self.n_win, self.tok_cap, self.n_cap = B, m, n_win, tok_cap, n_cap
        self.ctx = np.zeros(B, dtype=np.int64) if ctx is None else np.asarray(ctx, np.int64).copy()
        if self.ctx.shape != (B,) or (self.ctx < 0).any():
            raise ValueError("ctx must hold B non-negative lengths")

    def complete_blocks(self) -> np.ndarray:
        """Complete blocks per sequence (entries the compressed cache can hold)."""
        return self.ctx // self.m

    def ring_tokens_needed(self, n_new) -> int:
        """Per-token slots an append of n_new tokens per sequence reads at once: the
        new queries' windows reach n_win - 1 tokens before the first new token, and
        the first block they complete starts up to m - 1 tokens before it."""
        n = int(np.max(np.asarray(n_new)))
        if n <= 0:
            return 0
        return n + max(self.n_win, self.m) - 1

    def slots(self, b: int, n_new: int) -> np.ndarray:
        """Slots of the per-token buffer where sequence b's next n_new tokens go."""
        return (self.ctx[b] + np.arange(n_new, dtype=np.int64)) % self.tok_cap

    def append(self, n_new):
        """Record n_new[b] new tokens per sequence; returns (blk_begin int32 [B],
        n_blk) for one compressor call, n_blk = 0 when no block completed."""
        n_new = np.asarray(n_new, dtype=np.int64).reshape(-1)
        if n_new.shape != (self.B,) or (n_new < 0).any():
            raise ValueError("n_new must hold B non-negative counts")
        need = self.ring_tokens_needed(n_new)
        if need > self.tok_cap:
            raise ValueError(f"tok_cap = {self.tok_cap} slots cannot hold the {need} tokens "
                             f"this append reads at once")
        before = self.ctx // self.m
        after = (self.ctx + n_new) // self.m
        if (after > self.n_cap).any():
            raise ValueError(f"n_cap = {self.n_cap} entries cannot hold {int(after.max())} blocks")
        done = after - before
        n_blk = int(done.max())
        blk_begin = np.where(done > 0, before, -1).astype(np.int32)
        self.ctx = self.ctx + n_new
        return blk_begin, n_blk

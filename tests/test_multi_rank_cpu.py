"""Two ranks on the CPU (gloo): the replica timing reduction of bench.py, and the
algebra of splitting one long sequence's compressed entries over ranks.

The decode batch shards by sequence with no exchange (replicas), so bench.py runs
one replica per rank and reports the job at the pace of its slowest rank.  A
single long sequence would shard its compressed entries: every rank scores its
range and keeps its local top k; the k candidates of every rank are gathered and
the global top k taken by (score descending, index ascending), which is the
sequence's exact top k because every member of it is in its own rank's local top
k; every rank attends to the selected entries of its range (the rank holding the
tail also to the window), and the (o, lse) partials are gathered and merged.
This file checks that algebra with the oracle against the one-process result.
"""
import math
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _timing_worker(rank, world, port, out):
    _init(rank, world, port)
    import bench
    ms = [3.0, 7.5][rank]
    out[rank] = bench.max_over_ranks(ms, "cpu", dist, world)
    dist.destroy_process_group()


def test_replica_timing_is_the_slowest_rank():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_timing_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 7.5


# one CSA decode query at small sizes (2,048 tokens, 8 heads of 64 dims)
L, D, H, H_I, D_I, M, N_WIN, K = 2048, 64, 8, 2, 32, 4, 128, 16


def _inputs():
    rng = np.random.default_rng(5)
    n = L // M
    ck = rng.standard_normal((n, D)) / math.sqrt(D)
    cv = rng.standard_normal((n, D)) / math.sqrt(D)
    cI = rng.standard_normal((n, D_I)) / math.sqrt(D_I)
    k_tok = rng.standard_normal((L, D)) / math.sqrt(D)
    v_tok = rng.standard_normal((L, D)) / math.sqrt(D)
    q = rng.standard_normal((H, D)) / math.sqrt(D)
    qI = rng.standard_normal((H_I, D_I)) / math.sqrt(D_I)
    w = rng.uniform(0, 1, H_I)
    return q, qI, w, ck, cv, cI, k_tok, v_tok


class OracleOps:
    """The local stages of long_context_hybrid_02_b300.sharded done by the oracle on
    the CPU (float64 tensors), so that the runtime's exchange (candidate packing,
    the all-gathers, the split of the selection) runs on gloo ranks without a GPU."""

    def __init__(self, k_tok, v_tok):
        self.k_tok, self.v_tok = k_tok, v_tok

    def candidates(self, sh, qI, w, t):
        from long_context_hybrid_02_b300 import sharded as S
        ctx = S.shard_ctx_len(t, sh.j0, sh.j1, N_WIN, M, 0)
        n_loc = O.n_eligible(ctx - 1, N_WIN, M)
        # the shard's eligibility is the global one restricted to its range
        assert n_loc == len([j for j in range(sh.j0, sh.j1) if j < O.n_eligible(t, N_WIN, M)])
        s = O.index_scores(qI, w, sh.cki[:n_loc])
        loc = torch.from_numpy(O.topk_select(s, K)).to(torch.int32)
        scores = torch.from_numpy(np.concatenate([s, np.zeros(max(0, sh.j1 - sh.j0 - n_loc))]))
        return S.pack_candidates(scores, loc, sh.j0)

    def select(self, p, cand_scores, cand_idx):
        pick = torch.from_numpy(O.topk_select(cand_scores.numpy(), K))
        g = cand_idx[pick.clamp(min=0)]
        return torch.where(pick >= 0, g, torch.full_like(g, -1)).to(torch.int32)

    def partial(self, sh, q, sel, t):
        from long_context_hybrid_02_b300 import sharded as S
        local = S.split_selection(sel, sh.j0, sh.j1).numpy()
        mine = local[local >= 0]
        keys, vals = sh.ck[mine], sh.cv[mine]
        if sh.k_tok is not None:
            win = O.window_positions(t, N_WIN)
            keys = np.concatenate([keys, self.k_tok[win]])
            vals = np.concatenate([vals, self.v_tok[win]])
        o, lse = O.attend(q, keys, vals, 1 / math.sqrt(D))
        return torch.from_numpy(o), torch.from_numpy(lse)

    def merge(self, p, o_parts, lse_parts, dtype):
        o, lse = O.merge_partials(o_parts.numpy(), lse_parts.numpy())
        return torch.from_numpy(o), torch.from_numpy(lse)


def _shard_worker(rank, world, port, out):
    _init(rank, world, port)
    from long_context_hybrid_02_b300 import sharded as S
    q, qI, w, ck, cv, cI, k_tok, v_tok = _inputs()
    n = L // M
    j0, j1 = S.shard_range(n, rank, world)
    tail = rank == world - 1
    sh = S.Shard(p=None, ck=ck[j0:j1], cv=cv[j0:j1], cki=cI[j0:j1], j0=j0, j1=j1,
                 k_tok=k_tok if tail else None, v_tok=v_tok if tail else None)
    o, lse, sel = S.sharded_decode(sh, q, qI, w, L - 1, world, ops=OracleOps(k_tok, v_tok))
    out[rank] = (sel.tolist(), o.numpy(), lse.numpy())
    dist.destroy_process_group()


def _run_sharded(world):
    out = mp.Manager().dict()
    mp.spawn(_shard_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    q, qI, w, ck, cv, cI, k_tok, v_tok = _inputs()
    o_ref, lse_ref, idx_ref, _ = O.csa_decode(q, qI, w, ck, cv, cI, k_tok, v_tok, L - 1,
                                              n_win=N_WIN, m=M, k=K, scale=1 / math.sqrt(D))
    for r in range(world):
        sel, o, lse = out[r]
        assert sorted(j for j in sel if j >= 0) == [int(j) for j in idx_ref if j >= 0]
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-14)


def test_sharded_long_sequence_equals_one_process_two_ranks():
    """The runtime's exchange over two gloo ranks (local stages by the oracle) gives
    the one-process oracle result."""
    _run_sharded(2)


def test_sharded_long_sequence_equals_one_process_three_ranks():
    """Three ranks: uneven ranges, the window on the last one."""
    _run_sharded(3)


def test_shard_eligibility_and_selection_split():
    """shard_ctx_len makes a shard's own eligibility equal to the global one on its
    range (both rules, counted by enumeration); split_selection keeps exactly the
    shard's entries; pack_candidates marks padding with -inf / -1."""
    from long_context_hybrid_02_b300 import sharded as S
    from long_context_hybrid_02_b300 import binding as B
    n = 100
    for rule, rname in ((B.ELIG_DISJOINT, "disjoint"), (B.ELIG_OVERLAP, "overlap")):
        for t in (0, 5, 127, 128, 131, 300, 527, 1000):
            ne = O.n_eligible(t, N_WIN, M, rname)
            for world in (1, 2, 3, 7):
                for r in range(world):
                    j0, j1 = S.shard_range(n, r, world)
                    ctx = S.shard_ctx_len(t, j0, j1, N_WIN, M, rule)
                    got = O.n_eligible(ctx - 1, N_WIN, M, rname)
                    assert got == sum(1 for j in range(j0, j1) if j < min(ne, n)), (t, world, r)
    sel = torch.tensor([3, 10, 11, 40, 99, -1], dtype=torch.int32)
    assert S.split_selection(sel, 10, 41).tolist() == [-1, 0, 1, 30, -1, -1]
    s, g = S.pack_candidates(torch.arange(50, dtype=torch.float32),
                             torch.tensor([2, 7, -1], dtype=torch.int32), 100)
    assert s.tolist()[:2] == [2.0, 7.0] and s[2] == float("-inf") and g.tolist() == [102, 107, -1]

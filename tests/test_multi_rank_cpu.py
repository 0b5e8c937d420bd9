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


def _shard_worker(rank, world, port, out):
    _init(rank, world, port)
    q, qI, w, ck, cv, cI, k_tok, v_tok = _inputs()
    t = L - 1
    ne = O.n_eligible(t, N_WIN, M)
    lo, hi = ne * rank // world, ne * (rank + 1) // world
    # local scores and local top k, as (score, global index) candidates
    s_loc = O.index_scores(qI, w, cI[lo:hi])
    loc = O.topk_select(s_loc, K)
    cand = np.full((K, 2), [-np.inf, -1.0])
    for i, j in enumerate(loc[loc >= 0]):
        cand[i] = (s_loc[j], lo + j)
    gathered = [torch.zeros(K, 2, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(cand))
    allc = torch.cat(gathered).numpy()
    allc = allc[allc[:, 1] >= 0]
    order = np.lexsort((allc[:, 1], -allc[:, 0]))         # score descending, then index
    sel = np.sort(allc[order[:K], 1].astype(np.int64))
    # attention partial over this rank's selected entries (+ the window on the last rank)
    mine = sel[(sel >= lo) & (sel < hi)]
    keys, vals = ck[mine], cv[mine]
    if rank == world - 1:
        win = O.window_positions(t, N_WIN)
        keys, vals = np.concatenate([keys, k_tok[win]]), np.concatenate([vals, v_tok[win]])
    o_r, lse_r = O.attend(q, keys, vals, 1 / math.sqrt(D))
    og = [torch.zeros(H, D, dtype=torch.float64) for _ in range(world)]
    lg = [torch.zeros(H, dtype=torch.float64) for _ in range(world)]
    dist.all_gather(og, torch.from_numpy(o_r))
    dist.all_gather(lg, torch.from_numpy(lse_r))
    o, lse = O.merge_partials(np.stack([x.numpy() for x in og]), np.stack([x.numpy() for x in lg]))
    out[rank] = (sel.tolist(), o, lse)
    dist.destroy_process_group()


def test_sharded_long_sequence_equals_one_process():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_shard_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    q, qI, w, ck, cv, cI, k_tok, v_tok = _inputs()
    o_ref, lse_ref, idx_ref, _ = O.csa_decode(q, qI, w, ck, cv, cI, k_tok, v_tok, L - 1,
                                              n_win=N_WIN, m=M, k=K, scale=1 / math.sqrt(D))
    for r in range(world):
        sel, o, lse = out[r]
        assert sel == [int(j) for j in idx_ref if j >= 0]
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-14)

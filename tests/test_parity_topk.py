"""csa_topk against the oracle's selection, bit-exact, in every launch configuration.

Rows of up to 40,960 entries go to one 1024-thread CTA each (keys in shared
memory, a sampled threshold, early stop of the digit passes).  Longer rows are
cut into segments of at most 40,960 keys: one CTA per segment keeps the keys at
or above a local sampled threshold, one CTA per row selects among them, and a
row whose selection could miss a key (or whose lists overflow) is selected again
from all of its scores.  The scores are fed identically to both sides
(float32), so the index sets must be identical: ties broken by the smaller
index, NaN ranked as -inf, output in ascending index order with -1 padding.
"""
import numpy as np
import pytest
import torch

import oracle as O
from long_context_hybrid_02_b300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(scores, q_pos, k, m=4, n_win=128):
    Bn, Tq, n_cap = scores.shape
    p = B.make_params(Bn, 1, 512, n_win, m, k, 1, 8, B.F32)
    idx = torch.full((Bn, Tq, k), -7, dtype=torch.int32, device=DEV)
    nb = B.ha_workspace_size(p, B.OP_TOPK, Tq, n_cap, True)
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV)
    B.csa_topk(p, scores.to(DEV), n_cap, q_pos.to(DEV), Tq, idx, (ws.data_ptr(), ws.numel()))
    torch.cuda.synchronize()
    return idx.cpu().numpy()


def _check(scores, q_pos, idx, k, m=4, n_win=128):
    Bn, Tq, n_cap = scores.shape
    for b in range(Bn):
        for t in range(Tq):
            ne = min(O.n_eligible(int(q_pos[b, t]), n_win, m), n_cap)
            ref = O.topk_select(scores[b, t, :ne].double().numpy(), k)
            assert idx[b, t].tolist() == ref.tolist(), (b, t, ne)


def _scores(shape, seed, ties=None, nans=0):
    g = torch.Generator().manual_seed(seed)
    s = torch.randn(shape, generator=g)
    if ties:
        s = torch.round(s * ties) / ties
    if nans:
        flat = s.view(-1)
        flat[torch.randperm(flat.numel(), generator=g)[:nans]] = float("nan")
    return s


def test_topk_million_token_rows_in_segments():
    """4 rows x 262,144 entries, k = 1024: segments of ~7K keys; heavy ties and an
    all-equal row overflow the segment lists and take the all-score path."""
    n_cap, k = 262144, 1024
    s = _scores((4, 1, n_cap), 1)
    s[1] = torch.round(s[1] * 8) / 8                        # heavy ties
    s[2, 0, ::7] = float("nan")
    s[3, 0, :] = 0.5                                        # all equal
    q_pos = torch.full((4, 1), 128 + 4 * n_cap - 1, dtype=torch.int32)
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)


def test_topk_long_rows_of_different_lengths():
    """Rows of 400,000 and 300,000 eligible entries with ties (many segments, the
    last one ragged)."""
    n_cap, k = 400000, 512
    s = _scores((2, 1, n_cap), 2, ties=16)
    q_pos = torch.tensor([[128 + 4 * n_cap - 1], [128 + 4 * 300000 - 1]], dtype=torch.int32)
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)


def test_topk_many_rows_one_cta_each_ragged_eligibility():
    """300 prefill rows (one CTA per row) with eligible counts from 0 to n_cap."""
    n_cap, k = 5000, 512
    rng = np.random.default_rng(3)
    ne = rng.integers(0, n_cap + 1, 300)
    ne[:4] = [0, 1, k, k + 1]
    q_pos = torch.tensor((128 + 4 * ne - 1).reshape(1, 300), dtype=torch.int32)
    q_pos[0, 0] = 5                                         # no eligible entry
    s = _scores((1, 300, n_cap), 4, ties=4, nans=3000)
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)


@pytest.mark.parametrize("n_cap,k", [(700, 512), (16384, 512), (33792, 512), (8192, 1024)])
def test_topk_decode_batches(n_cap, k):
    s = _scores((32, 1, n_cap), 5 + n_cap, ties=32, nans=50)
    q_pos = torch.full((32, 1), 128 + 4 * n_cap - 1, dtype=torch.int32)
    q_pos[5, 0] = 128 + 4 * (k - 3) - 1                     # fewer eligible than k
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)


def test_topk_signed_zeros_tie():
    """-0.0 and +0.0 are one score: the tie goes to the smaller index."""
    n_cap, k = 2048, 512
    s = torch.zeros((2, 1, n_cap))
    s[0, 0, ::2] = -0.0                                     # alternate -0 / +0, all tied
    s[1, 0, :300] = 1.0
    s[1, 0, 300::3] = -0.0                                  # threshold at zero
    q_pos = torch.full((2, 1), 128 + 4 * n_cap - 1, dtype=torch.int32)
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)
    assert idx[0, 0].tolist() == list(range(k))


@pytest.mark.parametrize("rows,n_cap", [(148, 10000), (80, 16384), (300, 9000)])
def test_topk_segments_near_the_default_shared_memory_limit(rows, n_cap):
    """Segments whose keys (plus the kernel's static shared memory) pass the 48 KiB
    default, with and without clusters."""
    k = 512
    s = _scores((1, rows, n_cap), 20 + rows, ties=8)
    q_pos = torch.full((1, rows), 128 + 4 * n_cap - 1, dtype=torch.int32)
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)


@pytest.mark.parametrize("n_cap", [40960, 40961])
def test_topk_largest_one_cta_row_and_first_cluster_row(n_cap):
    """The last row length held by one CTA, and the first one split over a cluster."""
    k = 1024
    s = _scores((3, 1, n_cap), 30, ties=64, nans=200)
    q_pos = torch.full((3, 1), 128 + 4 * n_cap - 1, dtype=torch.int32)
    q_pos[2, 0] = 128 + 4 * (n_cap - 37) - 1                # ragged: not a multiple of 32
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)


def test_topk_one_cta_all_equal_and_threshold_ties():
    """Every digit pass runs to the end: the whole row, or a large share of it, ties
    at the threshold, and the ties are taken by index."""
    n_cap, k = 20000, 512
    s = torch.full((4, 1, n_cap), 0.25)
    s[1, 0, 5000:5100] = 3.0                                 # 100 above, the rest tied
    s[2, 0, ::3] = float("nan")                              # NaN below every tie
    s[3, 0, 19000:] = torch.arange(1000, dtype=torch.float32) # distinct top, ties below
    q_pos = torch.full((4, 1), 128 + 4 * n_cap - 1, dtype=torch.int32)
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)
    assert idx[0, 0].tolist() == list(range(k))


def test_topk_one_cta_bin_taken_whole():
    """The k largest keys sit alone in the top first-digit bins: the passes stop
    after the first one."""
    n_cap, k = 9000, 512
    g = torch.Generator().manual_seed(31)
    s = torch.rand((2, 1, n_cap), generator=g)               # [0, 1)
    pick = torch.randperm(n_cap, generator=g)[:k]
    s[0, 0, pick] = 1e6                                      # one bin holds exactly k keys
    s[1, 0, pick] = 1e6 + torch.arange(k, dtype=torch.float32) * 64
    q_pos = torch.full((2, 1), 128 + 4 * n_cap - 1, dtype=torch.int32)
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)
    assert sorted(pick.tolist()) == idx[0, 0].tolist()


def test_topk_one_cta_sample_blind_rows():
    """Rows whose large scores sit where the strided threshold sample never looks
    (period 16 at phase 3), and rows of fewer than 4,096 keys that all tie: the
    kernel's sampled threshold misjudges them and the exact passes over every key
    take over."""
    n_cap, k = 16384, 512
    g = torch.Generator().manual_seed(32)
    s = torch.rand((3, 1, n_cap), generator=g)
    s[0, 0, 3::16] += 5.0                                    # 1,024 large keys, unseen by the sample
    s[1, 0, 3::16] += torch.rand(1024, generator=g) * 5.0
    s[2, 0, :] = 1.0
    q_pos = torch.full((3, 1), 128 + 4 * n_cap - 1, dtype=torch.int32)
    q_pos[2, 0] = 128 + 4 * 3000 - 1                         # 3,000 tied keys
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)


def test_topk_long_rows_with_the_top_in_few_segments():
    """The top k of a long row sits in its first tenth (so the first segments'
    local thresholds are too high and the row is selected from all its scores),
    or is planted in 1 % of the entries spread over the row (the sampled path)."""
    n_cap, k = 150000, 1024
    g = torch.Generator().manual_seed(33)
    s = torch.randn((2, 1, n_cap), generator=g)
    s[0, 0, : n_cap // 10] += 3.0
    s[1, 0, torch.randperm(n_cap, generator=g)[: n_cap // 100]] += 3.0
    q_pos = torch.full((2, 1), 128 + 4 * n_cap - 1, dtype=torch.int32)
    idx = _run(s, q_pos, k)
    _check(s, q_pos, idx, k)

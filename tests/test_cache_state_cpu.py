"""Host bookkeeping of the caches (CPU): after any sequence of ragged appends,
every complete block was last compressed by an append that came after it was
complete, compressor calls never reach past the compressed cache, blocks that
were compressed before they were complete are never eligible to a query of that
step, and a ring too small for an append is refused."""
import numpy as np
import pytest

import oracle as O
from long_context_hybrid_02_b300.cache_state import CacheState


def _simulate(B, m, n_win, tok_cap, n_cap, appends):
    st = CacheState(B, m, n_win, tok_cap, n_cap)
    last_done = {}                     # (b, j) -> length of sequence b when j was last compressed
    for n_new in appends:
        begin, n_blk = st.append(n_new)
        for b in range(B):
            if begin[b] < 0:
                continue
            for j in range(int(begin[b]), min(int(begin[b]) + n_blk, n_cap)):
                last_done[(b, j)] = int(st.ctx[b])
        # every query of this append sees only blocks that are complete now
        for b in range(B):
            lo = int(st.ctx[b]) - int(n_new[b])
            for t in range(lo, int(st.ctx[b])):
                ne = O.n_eligible(t, n_win, m)
                for j in range(ne):
                    assert (j + 1) * m <= int(st.ctx[b])
                    assert last_done[(b, j)] >= (j + 1) * m, (b, j)
    for b in range(B):
        for j in range(int(st.ctx[b]) // m):
            assert last_done[(b, j)] >= (j + 1) * m, (b, j)   # compressed once complete
    return st


@pytest.mark.parametrize("m", [4, 128])
def test_ragged_prefill_chunks_then_decode(m):
    rng = np.random.default_rng(m)
    B, n_win = 5, 128
    appends = [rng.integers(0, 700, B) for _ in range(4)] + [np.ones(B, np.int64)] * 300
    total = int(np.sum(appends, axis=0).max())
    st = _simulate(B, m, n_win, 4096, total // m + 1, appends)
    assert (st.ctx == np.sum(appends, axis=0)).all()


def test_decode_in_a_ring_of_window_size():
    # one token per step: a ring of max(n_win, m) slots is enough
    B, m, n_win = 3, 4, 128
    st = _simulate(B, m, n_win, 128, 1000, [np.ones(B, np.int64)] * 900)
    assert (st.complete_blocks() == 900 // m).all()


def test_blk_begin_marks_sequences_without_a_new_block():
    st = CacheState(3, 4, 128, 1024, 100, ctx=[3, 4, 6])
    begin, n_blk = st.append([1, 1, 1])          # lengths 4, 5, 7: only sequence 0 completes
    assert begin.tolist() == [0, -1, -1] and n_blk == 1 and begin.dtype == np.int32
    begin, n_blk = st.append([0, 0, 0])
    assert begin.tolist() == [-1, -1, -1] and n_blk == 0
    begin, n_blk = st.append([9, 3, 1])          # 13, 8, 8: blocks 1..2, 1, 1
    assert begin.tolist() == [1, 1, 1] and n_blk == 2


def test_slots_wrap_around_the_ring():
    st = CacheState(1, 4, 8, 16, 100, ctx=[14])
    assert st.slots(0, 4).tolist() == [14, 15, 0, 1]


def test_a_ring_too_small_for_the_append_is_refused():
    st = CacheState(1, 4, 128, 200, 1000, ctx=[1000])
    assert st.ring_tokens_needed([73]) == 200
    st.append([73])                               # exactly fits
    with pytest.raises(ValueError, match="tok_cap"):
        st.append([74])
    big = CacheState(1, 128, 128, 255, 1000)
    with pytest.raises(ValueError, match="tok_cap"):
        big.append([129])                         # 129 + 127 = 256 slots needed


def test_compressed_cache_capacity_is_checked():
    st = CacheState(2, 4, 128, 4096, 10)
    st.append([40, 12])
    with pytest.raises(ValueError, match="n_cap"):
        st.append([4, 0])                        # 44 tokens = 11 blocks


def test_bad_arguments():
    with pytest.raises(ValueError):
        CacheState(0, 4, 128, 128, 10)
    with pytest.raises(ValueError):
        CacheState(2, 4, 128, 128, 10, ctx=[1])
    st = CacheState(2, 4, 128, 128, 10)
    with pytest.raises(ValueError):
        st.append([1, -1])

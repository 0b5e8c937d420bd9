"""Plain CPU oracle of the hybrid long-context attention path (SWA + CSA / SWA + HCA).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` may import this module.  The CUDA library never calls it,
and it shares no code with the CUDA library: it imports numpy and the standard
library, nothing else.

Every function works on ONE sequence, in float64, on numpy arrays indexed by
absolute token position (no ring buffers, no blocking, no fusion).  Inputs may be
float32 or bfloat16-valued arrays; they are widened to float64 exactly.

Sources (web pages about DeepSeek-V4; none prints a formula, they give the data
flow and the constants):
  [V4-notes]  "DeepSeek-V4 深度研究剖析" (group-reading-wiki, DeepSeek-V4 research notes),
              §5.2 SWA (n_win = 128 uncompressed KV), §5.3 CSA (every m = 4 tokens'
              KV compressed into one entry; a Lightning Indexer scores the compressed
              entries and the top-k are attended; k = 512 Flash / 1024 Pro),
              §5.4 HCA (every m' = 128 tokens compressed into one entry, all
              attended densely), §5.5 (the three paths as one memory hierarchy),
              §8 (precision), §11.3 (deterministic kernels), §11.4 (cache kinds).
  [LateTalk]  "163: DeepSeek V4 Explained: The Infra Whale, 1M-Token Context Made
              Real, and Extreme Efficiency Optimization" (zjai.club), §14 (every
              layer is SWA plus one of CSA / HCA, fixed per layer; MQA-style shared KV).
  [EP95]      "EP 95 解读 DeepSeek-V4 论文" (aifrontier.kr), segment "处理 KV cache 的
              Lightning Indexer 与 top-k 选择" (compress first, the indexer looks at
              every compressed entry, take the top k, attend only to those) and the
              description of the attention-block figure (the uncompressed window and
              the compressed entries are concatenated before one MQA).

The pages leave the compressor and the indexer open.  The definitions used here
(and on the GPU) are:
  compressor : per block, softmax over the block's m scalar gate logits, then the
               gate-weighted sum of the block's rows (K, V and the indexer keys).
  indexer    : s_j = sum_h w_h * max(0, qI_h . cI_j).
Readings where the pages are silent (all listed with reasons in the design notes
of the repository):
  * eligibility: a compressed entry j is visible to the query at position t only
    when its whole block lies before the window ("disjoint"):
    n_elig(t) = floor(max(0, t + 1 - n_win) / m); the alternative "overlap" rule
    floor((t + 1) / m) is available as a flag.
  * the window of query t is the n_win positions max(0, t-n_win+1) .. t.
  * the window keys and the attended compressed entries share one softmax.
  * softmax scale 1/sqrt(d) over all d dims unless given.
  * top-k order: score descending, then smaller index; NaN scores rank as -inf;
    the result is emitted in ascending index order, padded with -1.
  * a query with no key at all (context 0) gives o = 0 and lse = -inf.
  * a given selection may hold entries that are not eligible: entries < 0 (the
    -1 padding) or >= min(n_elig(t), n_cap), n_cap = the rows of the compressed
    cache, are ignored; an entry listed twice is attended twice (the top-k never
    lists one twice).
  * compressed entries are rounded to the storage type (round-to-nearest-even to
    bfloat16, or to float32) because the cache stores them in that type.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "round_to_bf16", "round_to_storage", "round_to_e4m3", "fp8_kv_encode", "fp8_kv_decode",
    "fp8_kv_pack", "fp8_kv_unpack",
    "round_to_e2m1", "fp4_encode", "fp4_decode", "fp4_pack", "fp4_unpack",
    "gate_softmax", "compress_block",
    "compress", "n_eligible", "window_positions", "index_scores", "topk_select",
    "attend", "merge_partials", "csa_decode", "hca_decode", "prefill_query",
]


# --------------------------------------------------------------------------
# storage rounding ([V4-notes] §8: the KV cache is stored in a narrow type)
# --------------------------------------------------------------------------
def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits (1 implicit + 7 stored) and float32's
    exponent range.  Written directly on the float64 value (no float32 step, which
    would round twice).  Values below the bfloat16 normal range are not expected
    here and are rounded with the same 8-bit rule (no subnormal handling).
    """
    x = np.asarray(x, dtype=np.float64)
    mant, expo = np.frexp(x)                     # x = mant * 2**expo, |mant| in [0.5, 1)
    q = np.rint(np.ldexp(mant, 8))               # 8 significant bits, rint = ties-to-even
    return np.ldexp(q, expo - 8)


def round_to_storage(x, storage: str):
    """Round to the cache storage type: 'bf16' or 'f32'."""
    if storage == "bf16":
        return round_to_bf16(x)
    if storage == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    raise ValueError(f"unknown storage type {storage!r}")


# --------------------------------------------------------------------------
# the deployed KV format ([V4-notes] §8: the KV cache keeps its RoPE dims in BF16
# and its other dims in FP8).  The page names the split, not the layout; the
# reading used here: a K or V row of d = 512 dims keeps dims 0..63 (the RoPE
# dims) as bfloat16 and stores dims 64..511 as float8 e4m3fn values with one
# float32 scale per group of 64 dims, scale = max|x| / 448 over the group (so the
# largest element maps to the largest e4m3 value), codes rounded to nearest,
# ties to even; a row takes 128 + 448 + 28 = 604 bytes instead of 1,024 (stored
# padded to 608: fp8_kv_pack / fp8_kv_unpack).  As for FP4 below, the decisions
# (amax / 448 and x / scale) are float32 divisions of the row's float32 values,
# the precision the kernels take them in.
# --------------------------------------------------------------------------
E4M3_MAX = 448.0            # 1.75 * 2**8, the largest finite e4m3fn value
FP8_ROPE_DIMS = 64
FP8_GROUP = 64


def round_to_e4m3(x):
    """Round float64 values to the nearest float8 e4m3fn value, ties to even.

    e4m3fn: sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinity.  Normal
    values (1 + M/8) * 2**(E-7) for E = 1..15 (E = 15, M = 7 is NaN), so 2**-6 ..
    448; subnormals k * 2**-9, k = 1..7.  Magnitudes that round above 448 give
    NaN, as does NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, expo = np.frexp(a)                        # a = mant * 2**expo, mant in [0.5, 1)
    e = np.maximum(expo - 1, -6)                 # exponent of the leading bit; subnormals share -6
    step = np.ldexp(1.0, e - 3)                  # spacing of the 3-bit mantissa grid
    q = np.rint(a / step) * step                 # rint: ties to the even grid point
    q = np.where(q > E4M3_MAX, np.nan, q)
    q = np.where(np.isnan(x), np.nan, q)
    return np.copysign(q, x)


def fp8_kv_encode(row):
    """One K or V row in the FP8 format: (RoPE dims as bf16 [64], e4m3 codes
    [448 // 64, 64] as float64 values, float32 scales [448 // 64])."""
    row = np.asarray(row, dtype=np.float64)
    rope = round_to_bf16(row[:FP8_ROPE_DIMS])
    rest = row[FP8_ROPE_DIMS:].reshape(-1, FP8_GROUP).astype(np.float32)
    scale32 = (np.abs(rest).max(axis=1) / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(scale32 > 0, scale32, np.float32(1.0)).astype(np.float32)
    codes = round_to_e4m3((rest / safe[:, None]).astype(np.float32))
    codes[scale32 == 0] = 0.0
    return rope, codes, scale32.astype(np.float64)


FP8_ROW_BYTES = 608


def fp8_kv_pack(rope, codes, scale):
    """The stored FP8 row: bytes [0, 128) the RoPE dims as bfloat16, [128, 576) the
    e4m3fn codes of dims 64..511, [576, 604) the 7 float32 scales, [604, 608) zero."""
    out = np.zeros(FP8_ROW_BYTES, dtype=np.uint8)
    r32 = np.asarray(rope, dtype=np.float64).astype(np.float32)     # exact: bf16 values
    out[:128] = (r32.view(np.uint32) >> 16).astype(np.uint16).view(np.uint8)
    out[128:576] = _e4m3_bits(np.asarray(codes, dtype=np.float64).reshape(-1))
    out[576:604] = np.asarray(scale, dtype=np.float64).astype(np.float32).view(np.uint8)
    return out


def fp8_kv_unpack(row):
    """Inverse of fp8_kv_pack: (rope [64], codes [7, 64], scale [7]) as float64."""
    row = np.asarray(row, dtype=np.uint8)
    rope = (row[:128].view(np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes = _e4m3_value(row[128:576]).reshape(-1, FP8_GROUP)
    scale = row[576:604].copy().view(np.float32).astype(np.float64)
    return rope, codes, scale


def fp8_kv_decode(rope, codes, scale):
    """The row a FP8-format entry stands for (float64): RoPE dims, then code * scale."""
    return np.concatenate([np.asarray(rope, np.float64),
                           (np.asarray(codes, np.float64) * np.asarray(scale, np.float64)[:, None]).reshape(-1)])


# --------------------------------------------------------------------------
# the indexer in FP4 ([V4-notes] §8: the lightning indexer's attention
# computation runs in FP4, and its index scores are kept as BF16).  The page
# names the precision, not the layout; the reading used here: a row of indexer
# queries or keys is cut into groups of 16 consecutive elements, each element an
# e2m1 value (sign, 2 exponent bits, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2,
# 3, 4, 6) with one e4m3 scale per group, scale = max|x| / 6 rounded to e4m3,
# codes rounded to nearest, ties to even, magnitudes above 6 saturating to 6.
# The quantization decisions (amax / 6 and x / scale) are taken in float32, the
# precision the kernels take them in, on the float32 values of the inputs, so
# that both sides decide alike on the same inputs; the rounding steps themselves
# are exact.  A row is stored as 80 bytes: 64 bytes of codes (element 2i in the
# low nibble), the 8 scales, 8 unused bytes (fp4_pack / fp4_unpack).
# --------------------------------------------------------------------------
E2M1_MAX = 6.0
FP4_GROUP = 16


def round_to_e2m1(x):
    """Nearest e2m1 value (ties to the even mantissa), saturating at +-6; NaN stays NaN.

    Below 2 the values are 0.5 apart, in [2, 4) 1 apart, from 4 on 2 apart.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    _, expo = np.frexp(a)                          # a = f * 2**expo, f in [0.5, 1)
    e = np.maximum(expo - 1, 0)                    # binade of a (0 for a < 2)
    step = np.ldexp(1.0, e - 1)
    q = np.minimum(np.rint(a / step) * step, E2M1_MAX)   # rint: ties to even
    q = np.where(np.isnan(x), np.nan, q)
    return np.copysign(q, x)


def fp4_encode(rows):
    """Rows [n, d] (d a multiple of 16) -> (codes [n, d/16, 16] e2m1 values,
    scales [n, d/16] e4m3 values); an all-zero group gets scale 0 and codes 0.
    The divisions are float32 divisions of the rows' float32 values."""
    rows = np.asarray(rows, dtype=np.float64)
    n, d = rows.shape
    g = rows.reshape(n, d // FP4_GROUP, FP4_GROUP).astype(np.float32)
    amax = np.abs(g).max(axis=-1)
    scale = round_to_e4m3((amax / np.float32(E2M1_MAX)).astype(np.float32))
    safe = np.where(scale > 0, scale, 1.0).astype(np.float32)
    quot = (g / safe[..., None]).astype(np.float32)
    codes = np.where(scale[..., None] > 0, round_to_e2m1(quot), 0.0)
    return codes, scale


def fp4_pack(codes, scale):
    """The 80-byte rows of the FP4 indexer format: [n, 80] uint8."""
    codes = np.asarray(codes, dtype=np.float64)
    scale = np.asarray(scale, dtype=np.float64)
    n = codes.shape[0]
    flat = codes.reshape(n, -1)
    mag = np.abs(flat)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    idx = np.searchsorted(grid, mag)
    if not np.array_equal(grid[idx], mag):
        raise ValueError("codes off the e2m1 grid")
    nib = (idx | np.where(np.signbit(flat), 8, 0)).astype(np.uint8)
    out = np.zeros((n, 80), dtype=np.uint8)
    out[:, :64] = nib[:, 0::2] | (nib[:, 1::2] << 4)
    out[:, 64:72] = _e4m3_bits(scale)
    return out


def fp4_unpack(rows):
    """Inverse of fp4_pack: (codes [n, 8, 16], scales [n, 8]) as float64 values."""
    rows = np.asarray(rows, dtype=np.uint8)
    n = rows.shape[0]
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    nib = np.empty((n, 128), dtype=np.uint8)
    nib[:, 0::2] = rows[:, :64] & 15
    nib[:, 1::2] = rows[:, :64] >> 4
    codes = np.where(nib & 8, -1.0, 1.0) * grid[nib & 7]
    return codes.reshape(n, 8, 16), _e4m3_value(rows[:, 64:72])


def _e4m3_bits(v):
    """e4m3fn bit patterns of values on the e4m3fn grid (finite, sign of zero kept)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    bits = np.zeros(v.shape, dtype=np.int64)
    nz = a > 0
    e = np.floor(np.log2(np.where(nz, a, 1.0))).astype(np.int64)
    sub = nz & (e < -6)
    norm = nz & ~sub
    bits = np.where(norm, ((e + 7) << 3) | np.rint((a / np.exp2(e) - 1.0) * 8).astype(np.int64), bits)
    bits = np.where(sub, np.rint(a / 2.0 ** -9).astype(np.int64), bits)
    if not np.array_equal(_e4m3_value(bits.astype(np.uint8)), a):
        raise ValueError("values off the e4m3 grid")
    return (bits | np.where(np.signbit(v), 128, 0)).astype(np.uint8)


def _e4m3_value(bits):
    """Values of e4m3fn bit patterns (no NaN pattern expected)."""
    b = np.asarray(bits, dtype=np.int64)
    e, mnt = (b >> 3) & 15, b & 7
    val = np.where(e == 0, mnt * 2.0 ** -9, (1.0 + mnt / 8.0) * np.exp2(e - 7.0))
    return np.where(b & 128, -val, val)


def fp4_decode(codes, scale):
    """Inverse of fp4_encode: rows [n, d] = codes * scale of their group."""
    codes = np.asarray(codes, dtype=np.float64)
    scale = np.asarray(scale, dtype=np.float64)
    return (codes * scale[..., None]).reshape(codes.shape[0], -1)


# --------------------------------------------------------------------------
# a1 / a2: the token compressor ([V4-notes] §5.3 CSA m=4, §5.4 HCA m'=128)
# --------------------------------------------------------------------------
def gate_softmax(g):
    """Softmax of one block's m gate logits (max-subtracted, float64)."""
    g = np.asarray(g, dtype=np.float64)
    e = np.exp(g - g.max())
    return e / e.sum()


def compress_block(rows, g):
    """One compressed entry: sum_i alpha_i * rows[i], alpha = softmax(g) over the block."""
    alpha = gate_softmax(g)
    return alpha @ np.asarray(rows, dtype=np.float64)


def compress(X, gate, m: int, j_begin: int, n_blk: int, storage: str | None = None):
    """Compress blocks j_begin .. j_begin+n_blk-1 of a per-token array X [L, dX].

    Block j covers positions j*m .. j*m+m-1 and must be complete.  Returns
    [n_blk, dX]; rounded to ``storage`` when given.
    """
    X = np.asarray(X)
    gate = np.asarray(gate)
    lo, hi = j_begin * m, (j_begin + n_blk) * m
    if hi > X.shape[0]:
        raise ValueError(f"block {j_begin + n_blk - 1} is not complete")
    # every block at once: the same per-block softmax-gated sum as compress_block
    g = np.asarray(gate[lo:hi], dtype=np.float64).reshape(n_blk, m)
    e = np.exp(g - g.max(axis=1, keepdims=True))
    alpha = e / e.sum(axis=1, keepdims=True)                      # [n_blk, m]
    rows = np.asarray(X[lo:hi], dtype=np.float64).reshape(n_blk, m, X.shape[1])
    out = np.einsum("bi,bid->bd", alpha, rows)
    return out if storage is None else round_to_storage(out, storage)


# --------------------------------------------------------------------------
# what a query at position t sees ([V4-notes] §5.2, §5.3, §5.4)
# --------------------------------------------------------------------------
def n_eligible(t: int, n_win: int, m: int, rule: str = "disjoint") -> int:
    """Number of compressed entries (0 .. n-1) visible to the query at position t."""
    if rule == "disjoint":
        return max(0, t + 1 - n_win) // m
    if rule == "overlap":
        return (t + 1) // m
    raise ValueError(rule)


def window_positions(t: int, n_win: int) -> np.ndarray:
    """Positions of the uncompressed sliding window of the query at position t."""
    return np.arange(max(0, t - n_win + 1), t + 1, dtype=np.int64)


# --------------------------------------------------------------------------
# a3: Lightning Indexer score ([V4-notes] §5.3; [EP95] indexer segment)
# --------------------------------------------------------------------------
def index_scores(qI, w, cI):
    """s_j = sum_h w_h * max(0, qI_h . cI_j) for every row j of cI.

    qI [H_I, d_I], w [H_I], cI [n, d_I] -> [n] float64.
    """
    qI = np.asarray(qI, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    cI = np.asarray(cI, dtype=np.float64)
    dots = cI @ qI.T                              # [n, H_I]
    return np.maximum(dots, 0.0) @ w


# --------------------------------------------------------------------------
# a4: top-k selection ([V4-notes] §5.3: k = 512 / 1024)
# --------------------------------------------------------------------------
def topk_select(scores, k: int) -> np.ndarray:
    """Indices of the k best scores, best = larger score, then smaller index.

    All entries are taken when there are at most k.  NaN ranks as -inf.
    Returns int64 [k] in ascending index order, padded with -1.
    """
    s = np.asarray(scores, dtype=np.float64).copy()
    s[np.isnan(s)] = -np.inf
    n = s.shape[0]
    take = min(k, n)
    order = np.lexsort((np.arange(n), -s))        # primary key -s, then the index
    chosen = np.sort(order[:take].astype(np.int64))
    out = np.full(k, -1, dtype=np.int64)
    out[:take] = chosen
    return out


# --------------------------------------------------------------------------
# a5 / a6: joint attention and the split merge ([EP95] figure description:
# window and compressed entries concatenated before one multi-query attention)
# --------------------------------------------------------------------------
def attend(q, keys, values, scale: float):
    """Multi-query attention of H query heads over one shared set of keys.

    q [H, d], keys [n, d], values [n, dv] -> (o [H, dv], lse [H]) with
    z = scale * q.key, p = softmax(z) over the n keys, o = sum p * value,
    lse = log sum exp z.  n = 0 gives o = 0, lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    keys = np.asarray(keys, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    H = q.shape[0]
    if keys.shape[0] == 0:
        return np.zeros((H, values.shape[1])), np.full(H, -np.inf)
    z = scale * (q @ keys.T)                      # [H, n]
    zmax = z.max(axis=1, keepdims=True)
    e = np.exp(z - zmax)
    denom = e.sum(axis=1, keepdims=True)
    p = e / denom
    return p @ values, (zmax + np.log(denom))[:, 0]


def merge_partials(o_parts, lse_parts):
    """Combine attention results over disjoint key subsets.

    o_parts [S, H, dv], lse_parts [S, H]:  LSE = log sum_s exp(lse_s),
    o = sum_s exp(lse_s - LSE) * o_s.  Parts with lse = -inf carry no weight.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    mx = lse_parts.max(axis=0)
    H = lse_parts.shape[1]
    o = np.zeros(o_parts.shape[1:])
    lse = np.full(H, -np.inf)
    for h in range(H):
        if not np.isfinite(mx[h]):
            continue
        wgt = np.exp(lse_parts[:, h] - mx[h])
        tot = wgt.sum()
        lse[h] = mx[h] + math.log(tot)
        o[h] = (wgt / tot) @ o_parts[:, h, :]
    return o, lse


def _joint_keys(comp_idx, ck, cv, k_tok, v_tok, t, n_win, tok_base=0):
    """Key and value rows of one query: the compressed entries comp_idx, then the
    window positions of t (row u - tok_base of k_tok / v_tok holds position u).
    Rows are picked first and widened to float64 after (widening is exact)."""
    win = window_positions(t, n_win) - tok_base
    if win.size and win[0] < 0:
        raise ValueError("the per-token rows do not cover the window")
    comp_idx = np.asarray(comp_idx, dtype=np.int64)
    k_tok, v_tok = np.asarray(k_tok), np.asarray(v_tok)
    keys = np.concatenate([np.asarray(ck)[comp_idx].reshape(-1, k_tok.shape[1]).astype(np.float64),
                           k_tok[win].astype(np.float64)], axis=0)
    vals = np.concatenate([np.asarray(cv)[comp_idx].reshape(-1, v_tok.shape[1]).astype(np.float64),
                           v_tok[win].astype(np.float64)], axis=0)
    return keys, vals


# --------------------------------------------------------------------------
# one layer for one query, in the pages' order: compress -> index -> top-k -> attend
# --------------------------------------------------------------------------
def csa_decode(q, qI, w, ck, cv, cI, k_tok, v_tok, t: int, *, n_win: int, m: int, k: int,
               scale: float, rule: str = "disjoint"):
    """SWA + CSA for the query at position t of one sequence.

    ck, cv, cI: the compressed caches (entries 0 .. n-1, already in storage type);
    k_tok, v_tok: per-token K, V indexed by absolute position (at least t+1 rows).
    Returns (o [H, dv], lse [H], idx [k] ascending with -1 padding, scores [n_elig]).
    """
    ne = n_eligible(t, n_win, m, rule)
    scores = index_scores(qI, w, np.asarray(cI)[:ne])
    idx = topk_select(scores, k)
    sel = idx[idx >= 0]
    keys, vals = _joint_keys(sel, ck, cv, k_tok, v_tok, t, n_win)
    o, lse = attend(q, keys, vals, scale)
    return o, lse, idx, scores


def hca_decode(q, ck, cv, k_tok, v_tok, t: int, *, n_win: int, m: int, scale: float,
               rule: str = "disjoint"):
    """SWA + HCA for the query at position t: every eligible entry plus the window."""
    ne = n_eligible(t, n_win, m, rule)
    keys, vals = _joint_keys(np.arange(ne), ck, cv, k_tok, v_tok, t, n_win)
    return attend(q, keys, vals, scale)


def prefill_query(q, idx, ck, cv, k_tok, v_tok, t: int, *, n_win: int, m: int, scale: float,
                  rule: str = "disjoint", tok_base: int = 0):
    """Attention of one query at position t over a given selection plus its window.

    Serves a decode query (t = context length - 1) as well as each query of a
    prefill chunk.  idx: this query's selected entries (CSA, in any order, -1
    padded) or None for HCA (all eligible entries).  Entries of idx that are < 0
    or >= min(n_elig(t), n_cap), n_cap = len(ck), are ignored.  Positions between
    the last eligible block and the window start are not attended (the window
    stays exactly n_win wide).  Row r of k_tok / v_tok holds position tok_base + r
    (0: indexed by absolute position).
    """
    n_cap = np.asarray(ck).shape[0]
    ne = min(n_eligible(t, n_win, m, rule), n_cap)
    if idx is None:
        sel = np.arange(ne)
    else:
        idx = np.asarray(idx, dtype=np.int64).reshape(-1)
        sel = idx[(idx >= 0) & (idx < ne)]
    keys, vals = _joint_keys(sel, ck, cv, k_tok, v_tok, t, n_win, tok_base)
    return attend(q, keys, vals, scale)

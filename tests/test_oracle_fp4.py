"""Pins of the oracle's FP4 indexer format ("DeepSeek-V4 深度研究剖析" §8: the
lightning indexer computes in FP4), independent of the oracle's own arithmetic:

* the e2m1 grid enumerated from its bit fields: every value rounds to itself,
  every midpoint between neighbours to the one with the even mantissa,
  magnitudes past 6 saturate;
* the format's error bound on whole rows: every element within a quarter of
  max(|x|, scale) of the input (half the spacing of its binade), the largest
  element of each group within 2^-4 of itself (the e4m3 rounding of its scale),
  every scale on the e4m3 grid, an all-zero group exact.

And a diagnostic of the formats the page names for the indexer (not a pin of the
oracle): on seeded Gaussian indexer inputs the top-k taken from BF16-rounded
scores, and from scores of FP4 queries and keys, against the exact top-k.
"""
import math

import numpy as np
import torch
import pytest

import oracle as O


def e2m1_grid():
    """All non-negative e2m1 values with their mantissa bit, ascending."""
    vals = []
    for E in range(4):
        for M in range(2):
            v = M / 2 if E == 0 else (1 + M / 2) * 2.0 ** (E - 1)
            vals.append((v, M))
    return sorted(vals)


def test_e2m1_grid_round_trips():
    grid = e2m1_grid()
    v = np.array([g for g, _ in grid])
    assert v.tolist() == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    np.testing.assert_array_equal(O.round_to_e2m1(v), v)
    np.testing.assert_array_equal(O.round_to_e2m1(-v), -v)


def test_e2m1_midpoints_round_to_even_mantissa():
    grid = e2m1_grid()
    for (lo, m_lo), (hi, m_hi) in zip(grid[:-1], grid[1:]):
        mid = (lo + hi) / 2
        assert O.round_to_e2m1(mid) == (lo if m_lo % 2 == 0 else hi), (lo, hi)
        assert O.round_to_e2m1(math.nextafter(mid, 0)) == lo
        assert O.round_to_e2m1(math.nextafter(mid, math.inf)) == hi


def test_e2m1_saturates_and_keeps_nan():
    out = O.round_to_e2m1(np.array([6.5, 7.0, 100.0, np.inf, -9.0, np.nan]))
    np.testing.assert_array_equal(out[:5], [6.0, 6.0, 6.0, 6.0, -6.0])
    assert np.isnan(out[5])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fp4_rows_error_bound(seed):
    rng = np.random.default_rng(60 + seed)
    rows = rng.standard_normal((8, 128)) / math.sqrt(128)
    rows[3, 16:32] = 0.0                                       # an all-zero group
    codes, scale = O.fp4_encode(rows)
    assert codes.shape == (8, 8, 16) and scale.shape == (8, 8)
    np.testing.assert_array_equal(O.round_to_e4m3(scale), scale)
    assert scale[3, 1] == 0.0 and (codes[3, 1] == 0.0).all()
    assert set(np.unique(np.abs(codes))) <= {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}
    dec = O.fp4_decode(codes, scale)
    g, dg = rows.reshape(8, 8, 16), dec.reshape(8, 8, 16)
    bound = np.maximum(np.abs(g), scale[..., None]) / 4 * (1 + 2.0 ** -20)
    assert (np.abs(dg - g) <= bound).all()
    j = np.argmax(np.abs(g), axis=-1)
    top, dtop = np.take_along_axis(g, j[..., None], -1), np.take_along_axis(dg, j[..., None], -1)
    assert (np.abs(dtop - top) <= 2.0 ** -4 * np.abs(top) * (1 + 2.0 ** -20)).all()


def test_pins_catch_ties_rounded_away_from_zero(monkeypatch):
    good = O.round_to_e2m1

    def away(x):
        x = np.asarray(x, dtype=np.float64)
        a = np.abs(x)
        _, expo = np.frexp(a)
        step = np.ldexp(1.0, np.maximum(expo - 1, 0) - 1)
        return np.copysign(np.minimum(np.floor(a / step + 0.5) * step, 6.0), x)

    monkeypatch.setattr(O, "round_to_e2m1", away)
    with pytest.raises(AssertionError):
        test_e2m1_midpoints_round_to_even_mantissa()
    assert good(2.5) == 2.0 and away(2.5) == 3.0


# ----------------------------------------------------------------- diagnostic
H_I, D_I = 64, 128


def _indexer_inputs(rng, n, planted_frac=0.0):
    qI = O.round_to_bf16(rng.standard_normal((H_I, D_I)) / math.sqrt(D_I))
    w = rng.uniform(0.0, 1.0, H_I)
    keys = rng.standard_normal((n, D_I)) / math.sqrt(D_I) / 2   # ~ a gated mean of 4 rows
    planted = np.array([], dtype=np.int64)
    if planted_frac:
        u = (w[:, None] * qI).sum(0)
        u /= np.linalg.norm(u)
        planted = rng.choice(n, int(round(planted_frac * n)), replace=False)
        keys[planted] += 3.0 / math.sqrt(D_I) * u
    return qI, w, O.round_to_bf16(keys), set(planted.tolist())


def _selections(qI, w, keys, k):
    exact = set(O.topk_select(O.index_scores(qI, w, keys), k).tolist())
    s = O.index_scores(qI, w, keys)
    bf16 = set(O.topk_select(O.round_to_bf16(s.astype(np.float32)), k).tolist())
    q4 = O.fp4_decode(*O.fp4_encode(qI))
    k4 = O.fp4_decode(*O.fp4_encode(keys))
    fp4 = set(O.topk_select(O.index_scores(q4, w, k4), k).tolist())
    return exact, bf16, fp4


def test_recall_of_the_indexer_formats_on_gaussian_scores():
    """16,352 entries, top-512 (the 64K decode row): BF16 scores keep ~98-99.6 % of
    the exact set, FP4 queries and keys ~86 % (unstructured scores: the set is
    decided by small margins)."""
    rng = np.random.default_rng(7)
    k = 512
    exact, bf16, fp4 = _selections(*_indexer_inputs(rng, 16352)[:3], k)
    r_bf16, r_fp4 = len(exact & bf16) / k, len(exact & fp4) / k
    print(f"recall: bf16 scores {r_bf16:.4f}, fp4 indexer {r_fp4:.4f}")
    assert r_bf16 >= 0.97 and r_fp4 >= 0.75


def test_recall_of_the_indexer_formats_with_a_planted_subset():
    """65,536 entries, 1 % planted at +3 sigma, top-256: every selection, exact or
    in either format, is planted blocks only; the formats swap planted blocks."""
    rng = np.random.default_rng(8)
    k = 256
    qI, w, keys, planted = _indexer_inputs(rng, 65536, 0.01)
    exact, bf16, fp4 = _selections(qI, w, keys, k)
    assert exact <= planted and bf16 <= planted and fp4 <= planted
    r_bf16, r_fp4 = len(exact & bf16) / k, len(exact & fp4) / k
    print(f"recall with a planted subset: bf16 scores {r_bf16:.4f}, fp4 indexer {r_fp4:.4f}")
    assert r_bf16 >= 0.97 and r_fp4 >= 0.85


def test_fp4_row_bytes_worked_example_and_round_trip():
    """The 80-byte row: element 2i in the low nibble (sign in bit 3, magnitude index
    into 0, .5, 1, 1.5, 2, 3, 4, 6), the 8 e4m3fn scales after the 64 code bytes."""
    codes = np.zeros((1, 8, 16))
    scale = np.zeros((1, 8))
    codes[0, 0, 0], codes[0, 0, 1] = 1.0, -6.0        # nibbles 2 and 8|7 -> byte 0xF2
    codes[0, 7, 15] = 0.5                             # element 127 -> high nibble of byte 63
    scale[0] = [1.0, 448.0, 2.0 ** -9, -2.0, 0.0, 0.75, 1.125, 240.0]
    row = O.fp4_pack(codes, scale)
    assert row.shape == (1, 80) and row.dtype == np.uint8
    assert row[0, 0] == 0xF2 and row[0, 63] == 0x10 and (row[0, 1:63] == 0).all()
    assert row[0, 64:72].tolist() == [0x38, 0x7E, 0x01, 0xC0, 0x00, 0x34, 0x39, 0x77]
    assert (row[0, 72:] == 0).all()
    c2, s2 = O.fp4_unpack(row)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scale)


def test_fp4_scale_bits_match_torch_float8():
    """The scale bytes are torch's float8_e4m3fn bit patterns of the same values."""
    rng = np.random.default_rng(9)
    v = O.round_to_e4m3(rng.standard_normal(4000) * np.exp2(rng.uniform(-8, 8, 4000)))
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    codes = np.zeros((len(v), 8, 16))
    scale = np.zeros((len(v), 8))
    scale[:, 0] = v
    assert np.array_equal(O.fp4_pack(codes, scale)[:, 64], ref)


def test_fp4_pack_round_trips_encoded_rows():
    rng = np.random.default_rng(10)
    rows = rng.standard_normal((64, 128)) / math.sqrt(128)
    codes, scale = O.fp4_encode(rows)
    c2, s2 = O.fp4_unpack(O.fp4_pack(codes, scale))
    assert np.array_equal(O.fp4_decode(c2, s2), O.fp4_decode(codes, scale))

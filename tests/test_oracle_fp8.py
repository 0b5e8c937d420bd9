"""Pins of the oracle's FP8 KV format ("DeepSeek-V4 深度研究剖析" §8: RoPE dims in
BF16, the other dims in FP8), independent of the oracle's own arithmetic:

* the e4m3fn grid enumerated from its bit fields: every finite value rounds to
  itself, every midpoint between neighbours rounds to the one with the even
  mantissa, values past the largest finite one give NaN;
* a library routine: torch's float32 -> float8_e4m3fn cast on in-range values;
* the format's error bound on whole rows: RoPE dims exactly bf16-rounded, every
  other dim within half a mantissa step (2**-4 relative, or 2**-10 * scale in
  the subnormal range) of the input, the largest element of a group exact up
  to the float32 rounding of its scale.
"""
import math

import numpy as np
import pytest
import torch

import oracle as O


def e4m3_grid():
    """All finite non-negative e4m3fn values with their mantissa field, ascending."""
    vals = []
    for E in range(16):
        for M in range(8):
            if E == 15 and M == 7:
                continue                                       # the NaN encoding
            v = M / 8 * 2.0 ** -6 if E == 0 else (1 + M / 8) * 2.0 ** (E - 7)
            vals.append((v, M))
    vals.sort()
    return vals


def test_e4m3_grid_round_trips():
    grid = e4m3_grid()
    assert len(grid) == 127 and grid[-1][0] == 448.0 and grid[1][0] == 2.0 ** -9
    v = np.array([g for g, _ in grid])
    np.testing.assert_array_equal(O.round_to_e4m3(v), v)
    np.testing.assert_array_equal(O.round_to_e4m3(-v), -v)


def test_e4m3_midpoints_round_to_even_mantissa():
    grid = e4m3_grid()
    for (lo, m_lo), (hi, m_hi) in zip(grid[:-1], grid[1:]):
        mid = (lo + hi) / 2
        want = lo if m_lo % 2 == 0 else hi
        assert O.round_to_e4m3(mid) == want, (lo, hi)
        assert O.round_to_e4m3(math.nextafter(mid, 0)) == lo
        assert O.round_to_e4m3(math.nextafter(mid, math.inf)) == hi


def test_e4m3_overflow_and_nan():
    out = O.round_to_e4m3(np.array([460.0, 464.0, 470.0, 480.0, 1e6, np.inf, np.nan]))
    assert out[0] == 448.0 and out[1] == 448.0                # 464 is a tie: 448 has M = 6
    assert np.isnan(out[2:]).all()


def test_e4m3_matches_torch_cast():
    rng = np.random.default_rng(40)
    mag = np.exp(rng.uniform(math.log(2.0 ** -12), math.log(447.0), 20000))
    x = (mag * rng.choice([-1.0, 1.0], mag.size)).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(O.round_to_e4m3(x.astype(np.float64)), ref)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_fp8_kv_row_error_bound(seed):
    rng = np.random.default_rng(50 + seed)
    row = rng.standard_normal(512) / math.sqrt(512)
    row[64 + 64 * 3:64 + 64 * 4] = 0.0                         # an all-zero group
    rope, codes, scale = O.fp8_kv_encode(row)
    assert rope.shape == (64,) and codes.shape == (7, 64) and scale.shape == (7,)
    np.testing.assert_array_equal(rope, O.round_to_bf16(row[:64]))
    dec = O.fp8_kv_decode(rope, codes, scale)
    rest, drest = row[64:].reshape(7, 64), dec[64:].reshape(7, 64)
    assert scale[3] == 0.0 and (drest[3] == 0.0).all()
    bound = np.maximum(2.0 ** -4 * np.abs(rest), 2.0 ** -10 * scale[:, None]) * (1 + 2.0 ** -20)
    assert (np.abs(drest - rest) <= bound).all()
    for g in range(7):
        if scale[g] > 0:
            j = np.argmax(np.abs(rest[g]))
            assert abs(drest[g, j] - rest[g, j]) <= 2.0 ** -22 * abs(rest[g, j])


def test_fp8_kv_constant_row():
    row = np.full(512, -0.0371)
    rope, codes, scale = O.fp8_kv_encode(row)
    assert (codes == -448.0).all()
    dec = O.fp8_kv_decode(rope, codes, scale)
    assert np.abs(dec[64:] - row[64:]).max() <= 2.0 ** -23 * 0.0371


def test_diagnostic_attention_over_fp8_rows():
    """Not a pin: what the format costs one decode row of attention (640 keys, 64
    heads x 512) on seeded Gaussian rows.  The rows themselves move by ~2.35 %
    normwise (the RoPE dims stay bf16), o by about as much (V's rounding passes
    straight through the convex combination), lse barely (K's rounding averages
    out inside each logit)."""
    rng = np.random.default_rng(70)
    d, H, n = 512, 64, 640
    K = O.round_to_bf16(rng.standard_normal((n, d)) / math.sqrt(d))
    V = O.round_to_bf16(rng.standard_normal((n, d)) / math.sqrt(d))
    q = O.round_to_bf16(rng.standard_normal((H, d)) / math.sqrt(d) * 8)

    def fp8(rows):
        return np.stack([O.fp8_kv_decode(*O.fp8_kv_encode(r)) for r in rows])

    o, lse = O.attend(q, K, V, 1 / math.sqrt(d))
    o8, lse8 = O.attend(q, fp8(K), fp8(V), 1 / math.sqrt(d))
    rel_rows = np.linalg.norm(fp8(V) - V) / np.linalg.norm(V)
    rel_o = np.linalg.norm(o8 - o) / np.linalg.norm(o)
    print(f"fp8 rows {rel_rows:.4f}, o {rel_o:.4f}, max lse shift {np.abs(lse8 - lse).max():.2e}")
    assert 0.01 < rel_rows < 0.04 and rel_o < 0.04 and np.abs(lse8 - lse).max() < 1e-3


def test_pins_catch_a_scale_for_the_wrong_e4m3_variant(monkeypatch):
    # 240 is the largest finite value of the "fnuz" e4m3 variant, not of e4m3fn
    import oracle.hybrid_attention as H
    monkeypatch.setattr(H, "E4M3_MAX", 240.0)
    with pytest.raises(AssertionError):
        test_fp8_kv_constant_row()


def test_fp8_row_bytes_worked_example_and_round_trip():
    """The 608-byte row: bf16 RoPE dims, e4m3fn codes, float32 scales, 4 zero bytes."""
    rope = np.zeros(64)
    rope[0], rope[63] = 1.0, -2.5                    # bf16 0x3F80, 0xC020
    codes = np.zeros((7, 64))
    codes[0, 0], codes[6, 63] = 448.0, -0.75         # e4m3fn 0x7E, 0xB4
    scale = np.array([1.0, 0.5, 0.0, 2.0 ** -20, 3.0, 1e-3, 7.25])
    row = O.fp8_kv_pack(rope, codes, scale)
    assert row.shape == (608,) and row.dtype == np.uint8
    assert row[0:2].tolist() == [0x80, 0x3F] and row[126:128].tolist() == [0x20, 0xC0]
    assert row[128] == 0x7E and row[575] == 0xB4 and (row[129:575] == 0).all()
    assert row[576:580].tolist() == [0, 0, 0x80, 0x3F]          # float32 1.0
    assert (row[604:] == 0).all()
    r2, c2, s2 = O.fp8_kv_unpack(row)
    assert np.array_equal(r2, rope) and np.array_equal(c2, codes)
    assert np.array_equal(s2, scale.astype(np.float32).astype(np.float64))


def test_fp8_pack_round_trips_encoded_rows():
    rng = np.random.default_rng(12)
    for _ in range(20):
        row = rng.standard_normal(512) / math.sqrt(512)
        enc = O.fp8_kv_encode(row)
        assert np.array_equal(O.fp8_kv_decode(*O.fp8_kv_unpack(O.fp8_kv_pack(*enc))),
                              O.fp8_kv_decode(*enc))

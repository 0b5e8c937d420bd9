"""Comparison helpers shared by the parity tests (tolerances of the build spec).

floating point : |gpu - ref| <= atol + rtol * |ref| elementwise
                 float32 storage:  rtol 1e-4, atol 1e-4 * max|ref|
                 bfloat16 storage: rtol 2e-2, atol 1e-2
top-k          : index sets identical except for candidates whose oracle score lies
                 within 1e-6 (relative) of the oracle's k-th score.
lse            : a float32 result in every configuration, so it is not held to the
                 bfloat16 output tolerance.  With bfloat16 storage the tensor-core
                 attention multiplies V by P = exp(z - m) rounded to bfloat16 and
                 normalises by the sum of those rounded values (reading c20); each
                 rounding moves a value by at most 2^-9 of itself, so the sum, and
                 hence exp(lse), moves by at most 2^-9 relative: |dlse| <= 2^-9.
                 Tolerance: twice that, 2^-8 absolute, plus 1e-5 relative for the
                 float32 dot products.  Float32 storage: the float32 tolerance above.
"""
import numpy as np
import torch

TOL = {"f32": (1e-4, None), "bf16": (2e-2, 1e-2)}


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(gpu, ref, dtype: str, what: str = ""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    rtol, atol = TOL[dtype]
    if atol is None:
        atol = 1e-4 * (np.abs(ref).max() if ref.size else 0.0)
    err = np.abs(gpu - ref)
    bad = err > atol + rtol * np.abs(ref)
    if bad.any():
        i = np.unravel_index(np.argmax(err - (atol + rtol * np.abs(ref))), ref.shape)
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} elements out of tolerance; "
                             f"worst at {i}: gpu={gpu[i]!r} ref={ref[i]!r} (rtol={rtol}, atol={atol})")


LSE_ATOL_BF16 = 2.0 ** -8


def assert_lse_close(gpu, ref, dtype: str, what: str = ""):
    """lse against the oracle: float32-level for float32 storage; for bfloat16
    storage 2^-8 absolute + 1e-5 relative (twice the bound from the bfloat16
    rounding of P).  -inf (no key) must match exactly."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (what, gpu.shape, ref.shape)
    inf = np.isneginf(ref)
    assert (np.isneginf(gpu) == inf).all(), f"{what}: -inf pattern differs"
    if dtype == "f32":
        assert_close(gpu[~inf], ref[~inf], "f32", what)
        return
    err = np.abs(gpu[~inf] - ref[~inf])
    lim = LSE_ATOL_BF16 + 1e-5 * np.abs(ref[~inf])
    if (err > lim).any():
        i = int(np.argmax(err - lim))
        raise AssertionError(f"{what}: {int((err > lim).sum())}/{err.size} lse values out of "
                             f"tolerance; worst gpu={gpu[~inf][i]!r} ref={ref[~inf][i]!r} "
                             f"(atol={LSE_ATOL_BF16}, rtol=1e-5)")


def kth_score(scores: np.ndarray, k: int) -> float:
    s = np.where(np.isnan(scores), -np.inf, scores)
    order = np.lexsort((np.arange(s.size), -s))
    return s[order[k - 1]]


def assert_topk_match(gpu_idx, ref_idx, ref_scores, k: int, what: str = ""):
    """Index sets equal up to candidates within 1e-6 relative of the k-th oracle score."""
    g = set(int(x) for x in np.asarray(gpu_idx) if x >= 0)
    r = set(int(x) for x in np.asarray(ref_idx) if x >= 0)
    assert len(g) == len(r), f"{what}: {len(g)} selected vs {len(r)}"
    if g == r:
        return
    assert len(ref_scores) > k, f"{what}: sets differ although every entry is selected"
    kth = kth_score(np.asarray(ref_scores, dtype=np.float64), k)
    band = 1e-6 * abs(kth)
    for j in g.symmetric_difference(r):
        assert abs(ref_scores[j] - kth) <= band, (
            f"{what}: entry {j} (score {ref_scores[j]!r}) differs outside the band around "
            f"the k-th score {kth!r}")


def assert_sorted_unique(idx_row, n_valid: int, k: int, what: str = ""):
    v = [int(x) for x in idx_row]
    take = min(k, n_valid)
    assert all(x >= 0 for x in v[:take]) and all(x == -1 for x in v[take:]), what
    assert v[:take] == sorted(set(v[:take])), what
    assert all(x < n_valid for x in v[:take]), what

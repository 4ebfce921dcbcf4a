"""The two-term E4M3 splits that the decode kernel uses, checked on the CPU against the
bounds its tolerance argument rests on (not against the kernel itself).

hi is the FP32 value cut to 4 significant bits (sign, exponent and the top three mantissa
bits); lo is the FP32 remainder. Both are then converted to E4M3 (OCP fn) with
round-to-nearest-even, here through torch's conversion, as the kernel packs them.
* Queries: hi truncates (bit mask 0xFFF00000); q * 2^e with max|q| * 2^e in [128, 256).
  For every BF16 value whose scaled magnitude is at least 2^-2, hi + lo reproduces it
  exactly.
* Probabilities: hi rounds to nearest (add 0x80000, then mask), so |lo| is at most half a
  unit of hi's last place; P' = 2^(x - m + 7) <= 2^8.75. For P' >= 2^-1 (lo then an E4M3
  normal or zero), |hi + lo - P'| <= 2^-9 * P'. Below, the error is absolute: at most
  2^-10 for P' in [2^-6, 2^-1) (lo subnormal) and at most 2^-9 below 2^-6 (hi subnormal
  too).
"""
import numpy as np
import torch


def _hi(x: np.ndarray) -> np.ndarray:
    return (x.astype(np.float32).view(np.uint32) & np.uint32(0xFFF00000)).view(np.float32)


def _hi_rn(x: np.ndarray) -> np.ndarray:
    return ((x.astype(np.float32).view(np.uint32) + np.uint32(0x80000)) & np.uint32(0xFFF00000)).view(np.float32)


def _e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).float().numpy()


def _split(x: np.ndarray, hi_fn=_hi) -> np.ndarray:
    hi = hi_fn(x)
    return _e4m3(hi).astype(np.float64) + _e4m3(x - hi).astype(np.float64)


def test_query_split_is_exact_for_every_bf16_in_range():
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) < 2.0 ** 100)]
    for e in range(-4, 5):  # any scale: the split only sees q * 2^e
        x = vals * np.float32(2.0 ** e)
        keep = (np.abs(x) >= 0.25) & (np.abs(x) < 256)
        x = x[keep]
        np.testing.assert_array_equal(_split(x), x.astype(np.float64))


def test_query_hi_term_is_e4m3_exact_in_range():
    x = np.exp2(np.random.default_rng(1).uniform(-2.0, 8.0, 100_000)).astype(np.float32)
    hi = _hi(x)
    np.testing.assert_array_equal(_e4m3(hi), hi)


def test_probability_split_error_bounds():
    rng = np.random.default_rng(0)
    x = np.exp2(rng.uniform(-14.0, 8.75, 4_000_000)).astype(np.float32)
    # every FP32 mantissa pattern of one binade at 2^-10 spacing, in each region
    grid = 1.0 + np.arange(1024, dtype=np.float32) / 1024
    x = np.concatenate([x] + [grid * np.float32(2.0 ** k) for k in (-12, -8, -4, -1, 1, 7)])
    xd = x.astype(np.float64)
    err = np.abs(_split(x, _hi_rn) - xd)
    top = xd >= 2.0 ** -1
    assert np.all(err[top] <= 2.0 ** -9 * xd[top]), float((err[top] / xd[top]).max())
    mid = (xd >= 2.0 ** -6) & ~top
    assert np.all(err[mid] <= 2.0 ** -10), float(err[mid].max())
    low = xd < 2.0 ** -6
    assert np.all(err[low] <= 2.0 ** -9), float(err[low].max())
    # the bounds are tight within a factor of two
    assert (err[top] / xd[top]).max() > 2.0 ** -10
    assert err[mid].max() > 2.0 ** -11 and err[low].max() > 2.0 ** -10
    # the rounded high term never leaves E4M3's range below 2^8.75
    assert _e4m3(_hi_rn(np.array([2.0 ** 8.75], np.float32)))[0] <= 448.0

"""The decode's per-head softmax numerics, emulated on the CPU from its constants.

This restates the kernel's scheme for one head (it is not the oracle and shares nothing
with it): scores x in log2 units arrive in tiles; the reference m is reset to the tile
max + kRescaleSlack when the tile max exceeds m + kRescaleMargin, or falls more than
kRescaleDrop below m (never lower than kRescaleFloor under the highest reference so far),
with O and l scaled by 2^(m_old - m_new); P' = 2^(x - m + kPBias) enters P.V as two E4M3
terms (FP32 rounded to 4 significant bits, then the remainder, each converted to E4M3
with round-to-nearest-even) while the row sum l adds the FP32 P'. The constants are read
from csrc/common.cuh, so a change there is checked against the same bounds.
"""
import os
import re

import numpy as np
import pytest
import torch

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "sparse_mla_paged_gb300", "csrc", "common.cuh")


def _const(name: str) -> float:
    m = re.search(rf"constexpr float {name} = ([0-9.]+)f;", open(HEADER).read())
    assert m, name
    return float(m.group(1))


BIAS, MARGIN, SLACK = _const("kPBias"), _const("kRescaleMargin"), _const("kRescaleSlack")
DROP, FLOOR = _const("kRescaleDrop"), _const("kRescaleFloor")
E4M3_MAX = 448.0
TOL_A = TOL_R = 1e-2


def _hi(x):
    """Round to 4 significant bits (round half up on the magnitude), as the kernel does."""
    b = x.astype(np.float32).view(np.uint32)
    return ((b + np.uint32(0x80000)) & np.uint32(0xFFF00000)).view(np.float32)


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def _emulate(x, v, tile):
    """Returns (output, largest P', resets after the first tile)."""
    m, mtop, o, l, pmax, resets = -np.inf, -np.inf, 0.0, 0.0, 0.0, 0
    for t0 in range(0, len(x), tile):
        xs, vs = x[t0:t0 + tile], v[t0:t0 + tile]
        tm = xs.max()
        m_new = m
        if tm > m + MARGIN or (tm < m - DROP and m > mtop - FLOOR):
            m_new = max(tm + SLACK, mtop - FLOOR)
        if m_new != m:
            a = 0.0 if m == -np.inf else 2.0 ** (m - m_new)
            o, l, m = o * a, l * a, m_new
            resets += t0 > 0
        mtop = max(mtop, m)
        pp = np.exp2(xs - m + BIAS).astype(np.float32)
        pmax = max(pmax, float(pp.max()))
        h = _hi(pp)
        o += ((_e4m3(h) + _e4m3(pp - h)) * vs).sum()
        l += pp.astype(np.float64).sum()
    return o / l, pmax, resets


def _exact(x, v):
    w = np.exp2(x - x.max())
    return (w * v).sum() / w.sum()


def _within(got, ref):
    return abs(got - ref) <= TOL_A + TOL_R * abs(ref)


@pytest.mark.parametrize("tile", [64, 128])
def test_probabilities_never_overflow_e4m3(tile):
    rng = np.random.default_rng(1)
    for _ in range(50):
        # rising scores: every tile's max just under the raise threshold of the one before
        steps = rng.uniform(0.0, MARGIN, 40)
        x = np.repeat(np.cumsum(steps), tile) + rng.uniform(-0.01, 0.0, 40 * tile)
        _, pmax, _ = _emulate(x, np.ones_like(x), tile)
        assert pmax < E4M3_MAX
    assert 2.0 ** (BIAS + MARGIN) < E4M3_MAX
    # the rounded high term of the largest P' is still an E4M3 value (448 = 1.75 * 2^8)
    assert float(_hi(np.array([2.0 ** (BIAS + MARGIN)], np.float32))[0]) <= E4M3_MAX


@pytest.mark.parametrize("tile", [64, 128])
def test_spread_tails_stay_well_inside_tolerance(tile):
    rng = np.random.default_rng(0)
    worst = 0.0
    for _ in range(100):
        x = rng.normal(-12.0, 4.0, 2048)
        x[0] = 0.0
        v = rng.uniform(-1.0, 1.0, 2048)
        worst = max(worst, abs(_emulate(x, v, tile)[0] - _exact(x, v)))
    assert worst < 2e-3


def test_flat_tail_under_a_first_tile_maximum():
    """One dominant token opens the first tile; 2047 equal scores 15 log2 units below it
    carry values whose weighted sum cancels the dominant one, so the reference is 0."""
    x = np.full(2048, -15.0)
    x[0] = 0.0
    v = np.ones(2048)
    v[0] = -2047 * 2.0 ** -15
    for tile in (64, 128):
        got, _, _ = _emulate(x, v, tile)
        assert abs(got - _exact(x, v)) <= 1e-2


@pytest.mark.parametrize("tile", [64, 128])
def test_flat_tail_sweep(tile):
    """Flat tails from 4 to 24 log2 units under the first token, in quarter steps (so tail
    probabilities that are not powers of two are covered), with tail values up to 4 and a
    dominant value that makes the reference cancel."""
    worst = 0.0
    for k in np.arange(4.0, 24.0, 0.25):
        x = np.full(2048, -k)
        x[0] = 0.0
        for vt in (1.0, 2.0, 4.0):
            v = np.full(2048, vt)
            v[0] = -vt * 2047 * 2.0 ** -k
            got, _, _ = _emulate(x, v, tile)
            ref = _exact(x, v)
            assert _within(got, ref), (k, vt, got, ref)
            worst = max(worst, abs(got - ref) / (TOL_A + TOL_R * abs(ref)))
    assert worst < 0.9


@pytest.mark.parametrize("tile", [64, 128])
def test_flat_tail_before_the_maximum(tile):
    """The same tails with the dominant token last: the reference rises once, at the end."""
    for k in (10.5, 14.0, 15.25, 17.0, 20.0):
        x = np.full(2048, -k)
        x[-1] = 0.0
        v = np.full(2048, 2.0)
        v[-1] = -2.0 * 2047 * 2.0 ** -k
        got, _, resets = _emulate(x, v, tile)
        assert _within(got, _exact(x, v)), (k, got)
        assert resets == 1


def test_deep_tail_does_not_overflow_the_accumulator():
    """A tail 200 log2 units under the maximum: the reference stops kRescaleFloor below its
    highest value, the tail carries no weight and nothing overflows."""
    x = np.full(1024, -200.0)
    x[0] = 0.0
    v = np.full(1024, 3.0)
    v[0] = 1.0
    got, _, _ = _emulate(x, v, 128)
    assert np.isfinite(got) and abs(got - 1.0) <= 1e-3
    # the largest rescaled value stays far inside FP32: P' of the maximum <= 2^(bias + floor + margin)
    assert BIAS + FLOOR + MARGIN + np.log2(448.0 * 8192) < 127

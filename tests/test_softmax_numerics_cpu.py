"""The decode's per-head softmax numerics, emulated on the CPU from its constants.

This restates the kernel's scheme for one head (it is not the oracle and shares nothing
with it): scores x in log2 units arrive in tiles; the reference max m is raised to the
tile max + kRescaleSlack only when a tile exceeds m + kRescaleMargin (O and l scaled by
2^(m_old - m_new)); P' = 2^(x - m + kPBias) enters P.V as two E4M3 terms (FP32 truncation
to 4 significant bits, then the remainder, each rounded to E4M3) while the row sum l adds
the FP32 P'. The constants are read from csrc/common.cuh, so a change there is checked
against the same bounds.
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
E4M3_MAX = 448.0


def _hi(x):
    return (x.astype(np.float32).view(np.uint32) & np.uint32(0xFFF00000)).view(np.float32)


def _e4m3(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def _emulate(x, v, tile):
    m, o, l, pmax = -np.inf, 0.0, 0.0, 0.0
    for t0 in range(0, len(x), tile):
        xs, vs = x[t0:t0 + tile], v[t0:t0 + tile]
        if xs.max() > m + MARGIN:
            m_new = xs.max() + SLACK
            a = 0.0 if m == -np.inf else 2.0 ** (m - m_new)
            o, l, m = o * a, l * a, m_new
        pp = np.exp2(xs - m + BIAS).astype(np.float32)
        pmax = max(pmax, float(pp.max()))
        h = _hi(pp)
        o += ((_e4m3(h) + _e4m3(pp - h)) * vs).sum()
        l += pp.astype(np.float64).sum()
    return o / l, pmax


def _exact(x, v):
    w = np.exp2(x - x.max())
    return (w * v).sum() / w.sum()


@pytest.mark.parametrize("tile", [64, 128])
def test_probabilities_never_overflow_e4m3(tile):
    rng = np.random.default_rng(1)
    for _ in range(50):
        # rising scores: every tile's max just under the raise threshold of the one before
        steps = rng.uniform(0.0, MARGIN, 40)
        x = np.repeat(np.cumsum(steps), tile) + rng.uniform(-0.01, 0.0, 40 * tile)
        _, pmax = _emulate(x, np.ones_like(x), tile)
        assert pmax < E4M3_MAX
    assert 2.0 ** (BIAS + MARGIN) < E4M3_MAX


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


@pytest.mark.xfail(strict=True, reason="P' below 2^-10 rounds to zero in both E4M3 terms: a flat tail "
                   "14-17 log2 units under a first-tile maximum is dropped (an open item of the design)")
def test_flat_tail_under_a_first_tile_maximum():
    x = np.full(2048, -15.0)
    x[0] = 0.0
    v = np.ones(2048)
    v[0] = -2047 * 2.0 ** -15          # the reference cancels to zero
    got, _ = _emulate(x, v, 128)
    assert abs(got - _exact(x, v)) <= 1e-2

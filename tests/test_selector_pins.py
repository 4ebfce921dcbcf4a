"""Pins of the oracle's selector (attend.rs module doc: the decode's input is a row of token
ids with -1 holes; decode_k.rs decode_k: top index_topk pools, row r only takes pools that
end at or before q_pos[r]).

Reading checked: pool p (positions p*kpool .. p*kpool + kpool - 1) is eligible when
(p + 1)*kpool - 1 <= q_pos; the topk eligible pools of highest score are taken, equal
scores going to the lower pool and NaN ranking below every number; the row lists the taken
pools in ascending position, kpool ids each, then -1.

The checks: a brute force written here with numpy's lexsort (a library sort) on random
inputs full of ties, NaNs and infinities; invariants (adding a constant to every score or
scaling them by a positive factor leaves the selection unchanged); closed forms (fewer
eligible pools than topk takes all of them; q_pos below the first pool's end gives an
all-hole row). Planted mistakes in a copy of the oracle must fail them.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")


def brute(scores, q_pos, kpool, topk):
    rows, n_pools = scores.shape
    out = np.full((rows, topk * kpool), -1, dtype=np.int32)
    for r in range(rows):
        elig = np.nonzero((np.arange(n_pools) + 1) * kpool - 1 <= q_pos[r])[0]
        s = scores[r, elig].astype(np.float64)
        nan = np.isnan(s)
        key = np.where(nan, 0.0, -s)                 # descending score
        order = np.lexsort((elig, key, nan))         # NaN last, then score, then pool index
        taken = np.sort(elig[order][:topk])
        ids = (taken[:, None] * kpool + np.arange(kpool)[None, :]).reshape(-1)
        out[r, :ids.size] = ids
    return out


def _inputs(seed, rows=6, n_pools=200):
    g = np.random.default_rng(seed)
    s = g.integers(-4, 5, size=(rows, n_pools)).astype(np.float32) * 0.5   # many ties
    s[g.random((rows, n_pools)) < 0.05] = np.nan
    s[g.random((rows, n_pools)) < 0.02] = np.inf
    s[g.random((rows, n_pools)) < 0.02] = -np.inf
    q = g.integers(-2, n_pools * 4 + 3, size=rows).astype(np.int32)
    q[0] = n_pools * 4 - 1
    return s, q


def _checks(lib) -> bool:
    ok = True
    for seed, kpool, topk in [(0, 4, 16), (1, 1, 7), (2, 8, 300), (3, 4, 1), (4, 2, 50)]:
        s, q = _inputs(seed)
        got = oracle.select_pools(s, q, kpool, topk, lib=lib)
        ok = ok and np.array_equal(got, brute(s, q, kpool, topk))
    # invariants on finite, distinct scores
    g = np.random.default_rng(9)
    s = g.normal(size=(4, 300)).astype(np.float32)
    q = np.array([1199, 700, 50, 1000], np.int32)
    base = oracle.select_pools(s, q, 4, 40, lib=lib)
    ok = ok and np.array_equal(oracle.select_pools(s + np.float32(100.0), q, 4, 40, lib=lib), base)
    ok = ok and np.array_equal(oracle.select_pools(s * np.float32(3.0), q, 4, 40, lib=lib), base)
    # closed forms
    few = oracle.select_pools(s, np.array([11, 11, 11, 11], np.int32), 4, 40, lib=lib)
    ok = ok and np.array_equal(few[:, :12], np.tile(np.arange(12), (4, 1))) and np.all(few[:, 12:] == -1)
    none = oracle.select_pools(s, np.array([2, -1, 0, 2], np.int32), 4, 40, lib=lib)
    ok = ok and np.all(none == -1)
    return bool(ok)


def test_selector_matches_brute_force_and_invariants():
    assert _checks(None)


MUTANTS = {
    "ties to the higher pool": ("return (x->pool > y->pool) - (x->pool < y->pool);",
                                "return (x->pool < y->pool) - (x->pool > y->pool);"),
    "ascending score": ("return x->score > y->score ? -1 : 1;", "return x->score > y->score ? 1 : -1;"),
    "NaN first": ("if (xn != yn) return xn - yn;", "if (xn != yn) return yn - xn;"),
    "eligibility off by one": ("(int64_t)(p + 1) * kpool - 1 <= (int64_t)q_pos[r]",
                               "(int64_t)(p + 1) * kpool - 1 < (int64_t)q_pos[r]"),
    "pool start instead of end": ("(int64_t)(p + 1) * kpool - 1 <= (int64_t)q_pos[r]",
                                  "(int64_t)p * kpool <= (int64_t)q_pos[r]"),
    "output in rank order": ("qsort(taken, (size_t)m, sizeof(int32_t), cmp_i32);", ""),
    "one too few": ("int32_t m = n < topk ? n : topk;", "int32_t m = n < topk ? n : topk - 1;"),
}


def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "m.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libm.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(path), "-lm"])
    return oracle._bind(str(so))


def test_unmutated_copy_passes(tmp_path):
    assert _checks(_build_mutant(tmp_path, "#define LATENT 512", "#define LATENT 512"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_selector_mutant_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, *MUTANTS[name])
    assert not _checks(lib), f"planted mistake {name!r} passed every pin"

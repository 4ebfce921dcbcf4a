"""Planted mistakes: each plausible slip in the oracle must fail one of its pins.

Every case copies oracle/dsa_oracle.c, applies one textual mutation (a dropped scale, a
wrong index, swapped operands, an off-by-one hole rule, a broken FP8 field), builds the
copy with gcc into a temporary directory and runs the same independent checks the pin
tests use (dense masked brute force, FP8 table vs torch, numpy unique). The real oracle
is never modified.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
from sparse_mla_paged_gb300 import workloads as wl
from test_oracle_pins import _fp8_bytes_to_f64, dense_masked

SRC = os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")

MUTANTS = {
    "dropped k_scale": ("J->k_scale * J->e4m3[krow[c]]", "J->e4m3[krow[c]]"),
    "dropped v_scale": ("J->v_scale * J->e4m3[vrow[c]]", "J->e4m3[vrow[c]]"),
    "dropped sm_scale": ("s[j] = J->sm_scale * dot;", "s[j] = dot;"),
    "page from id % bs": ("+ id / J->block_size;", "+ id % J->block_size;"),
    "slot from id / bs": ("(int64_t)(id % J->block_size) * LATENT", "(int64_t)(id / J->block_size) * LATENT"),
    "V read from K": ("J->v_cache + off[j]", "J->k_cache + off[j]"),
    "no normalisation": ("o[c] /= z;", "o[c] /= 1.0;"),
    "duplicates kept": ("if (u == 0 || ids_out[u - 1] != ids_out[j])", "if (1)"),
    "hole bound off by one": ("id >= 0 && id < seq_len", "id >= 0 && id <= seq_len"),
    "block-table row ignored": ("(int64_t)seq * J->max_blocks_per_seq", "(int64_t)0 * J->max_blocks_per_seq"),
    "e4m3 bias 8": ("ldexp(1.0 + (double)mantissa / 8.0, exponent - 7)",
                    "ldexp(1.0 + (double)mantissa / 8.0, exponent - 8)"),
    "e4m3 subnormal scale": ("ldexp((double)mantissa / 8.0, 1 - 7)", "ldexp((double)mantissa / 8.0, 0 - 7)"),
    "softmax sign": ("double w = exp(s[j] - m);", "double w = exp(m - s[j]);"),
    "q head/row transposed": ("((int64_t)r * J->num_q_heads + h) * LATENT", "((int64_t)h * J->num_q_heads + r) * LATENT"),
    "row-to-sequence map": ("int32_t seq = r / J->rows_per_seq;", "int32_t seq = r % J->rows_per_seq;"),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name!r} not unique/found"
    path = tmp_path / "m.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libm.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o",
                           str(so), str(path), "-lm"])
    return oracle._bind(str(so))


def _cases():
    return [
        wl.tiny(),
        wl.random_case(num_seqs=3, rows_per_seq=2, heads=3, seq_lens=[100, 130, 64, 65, 190, 5],
                       block_size=8, sel_width=40, out_of_range_frac=0.1, dup_frac=0.2, seed=21),
        wl.random_case(split_kv=True, heads=2, seq_len=90, block_size=16, sel_width=30,
                       k_scale=0.07, v_scale=0.03, seed=22),
    ]


def _pins_pass(lib) -> bool:
    table = oracle.e4m3_table(lib=lib)
    ref = _fp8_bytes_to_f64(np.arange(256, dtype=np.uint8))
    ok = np.array_equal(np.isnan(table), np.isnan(ref)) and np.array_equal(
        table[~np.isnan(ref)], ref[~np.isnan(ref)])
    rng = np.random.default_rng(3)
    sel = rng.integers(-3, 120, size=(6, 50)).astype(np.int32)
    lens = rng.integers(0, 130, size=6).astype(np.int32)
    ids, cnt = oracle.resolve_indices(sel, lens, lib=lib)
    for r in range(6):
        want = np.unique(sel[r][(sel[r] >= 0) & (sel[r] < lens[r])])
        ok = ok and cnt[r] == want.size and np.array_equal(ids[r, :cnt[r]], want)
    for w in _cases():
        try:
            got = oracle.decode_workload(w, lib=lib)
        except ValueError:
            return False
        ok = ok and np.allclose(got, dense_masked(w), rtol=1e-12, atol=1e-12)
    return bool(ok)


def test_unmutated_copy_passes(tmp_path):
    lib = _build_mutant(tmp_path, "identity", "#define LATENT 512", "#define LATENT 512")
    assert _pins_pass(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    assert not _pins_pass(lib), f"planted mistake {name!r} passed every pin"

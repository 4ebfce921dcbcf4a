"""Pins for the CPU oracle: each checks it against something other than itself.

* FP8 decode: every code against torch.float8_e4m3fn (a library routine) and against
  values of the OCP FP8 table (tests/golden/e4m3_ocp_values.txt).
* Decode: against a dense masked brute force written here independently (numpy + torch's
  FP8 decode, a mask over *every* position 0..L-1 with set membership of the selected
  ids, one matmul), which attend.rs's module doc states is exactly equivalent.
* Closed forms: a hand-derived two-token example, single selected token, all holes,
  zero query, dominant score.
* Invariants: permuting, duplicating ids, adding holes or out-of-range ids.
* Index resolution: numpy's unique on the filtered row, and brute-force set equality.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from sparse_mla_paged_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------------
# Independent brute force (shares nothing with oracle/).
# ---------------------------------------------------------------------------------

def _fp8_bytes_to_f64(b: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(b, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def _bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def dense_masked(w, rows=None):
    """softmax over all positions < L with -inf where the position is not a selected id."""
    h = w.host()
    q = _bf16_bits_to_f64(h["q_bits"])
    kc = h["k_cache"].reshape(-1)
    vc = kc if h["v_cache"] is None else h["v_cache"].reshape(-1)
    bt = h["block_tables"].reshape(-1)
    lens = h["seq_lens"].reshape(-1)
    sel = h["sel_indices"]
    rows = range(w.rows) if rows is None else rows
    outs = []
    for r in rows:
        seq = r // w.rows_per_seq
        L = int(lens[r])
        out = np.zeros((w.num_q_heads, 512))
        if L > 0:
            pos = np.arange(L)
            pages = bt[seq * w.max_blocks_per_seq + pos // w.block_size].astype(np.int64)
            base = pages * w.cache_stride_bytes + (pos % w.block_size) * 512
            idx = base[:, None] + np.arange(512)[None, :]
            K = w.k_scale * _fp8_bytes_to_f64(kc[idx])
            V = w.v_scale * _fp8_bytes_to_f64(vc[idx])
            member = np.zeros(L, dtype=bool)
            for i in set(int(x) for x in sel[r]):
                if 0 <= i < L:
                    member[i] = True
            if member.any():
                s = w.sm_scale * (q[r] @ K.T)                 # [H, L]
                s = np.where(member[None, :], s, -np.inf)
                s = s - s.max(axis=1, keepdims=True)
                p = np.exp(s)
                out = (p @ V) / p.sum(axis=1, keepdims=True)
        outs.append(out)
    return np.stack(outs)


def _assert_close(a, b, rtol=1e-12, atol=1e-12):
    np.testing.assert_allclose(a, b, rtol=rtol, atol=atol)


# ---------------------------------------------------------------------------------
# Element decoding.
# ---------------------------------------------------------------------------------

def test_e4m3_table_matches_torch(oracle_mod):
    ours = oracle_mod.e4m3_table()
    ref = _fp8_bytes_to_f64(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF
    np.testing.assert_array_equal(ours[~nan], ref[~nan])
    # signed zero is kept
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_table_matches_ocp_values(oracle_mod):
    ours = oracle_mod.e4m3_table()
    n = 0
    with open(os.path.join(GOLDEN, "e4m3_ocp_values.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            code, val = line.split()
            code = int(code, 16)
            if val == "nan":
                assert math.isnan(ours[code])
            else:
                assert ours[code] == float(val), hex(code)
                assert math.copysign(1.0, ours[code]) == math.copysign(1.0, float(val))
            n += 1
    assert n >= 10


def test_bf16_decode_matches_torch(oracle_mod):
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 1 << 16, size=200, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]  # drop inf/nan patterns
    np.testing.assert_array_equal(oracle_mod.bf16_to_f64(bits), _bf16_bits_to_f64(bits))


# ---------------------------------------------------------------------------------
# Index resolution.
# ---------------------------------------------------------------------------------

def test_resolve_matches_numpy_unique(oracle_mod):
    rng = np.random.default_rng(2)
    rows, width = 40, 97
    sel = rng.integers(-5, 300, size=(rows, width)).astype(np.int32)
    sel[rng.random((rows, width)) < 0.2] = -1
    sel[3] = -1                                   # an all-hole row
    lens = rng.integers(0, 320, size=rows).astype(np.int32)
    lens[5] = 0                                   # an empty sequence
    ids, counts = oracle_mod.resolve_indices(sel, lens)
    for r in range(rows):
        row = sel[r]
        want = np.unique(row[(row >= 0) & (row < lens[r])])
        assert counts[r] == want.size
        np.testing.assert_array_equal(ids[r, :want.size], want)
        assert np.all(ids[r, want.size:] == -1)
        # brute-force set equality
        assert set(ids[r, :counts[r]].tolist()) == {int(x) for x in row if 0 <= x < lens[r]}
    assert counts[3] == 0 and counts[5] == 0


# ---------------------------------------------------------------------------------
# Decode vs the dense masked brute force.
# ---------------------------------------------------------------------------------

def test_tiny_config_matches_dense_masked(oracle_mod):
    w = wl.tiny()
    _assert_close(oracle_mod.decode_workload(w), dense_masked(w))


@pytest.mark.parametrize("kw", [
    dict(),
    dict(heads=3, seq_len=200, block_size=16, sel_width=50, hole_frac=0.2, dup_frac=0.1),
    dict(num_seqs=3, rows_per_seq=2, seq_lens=[100, 130, 64, 65, 190, 5], block_size=8,
         sel_width=40, out_of_range_frac=0.1),
    dict(split_kv=True, stride_pad=48, block_size=5, seq_len=77, sel_width=30),
    dict(shared_table=True, num_seqs=2, seq_len=96, block_size=32, sel_width=20),
    dict(cache_dist="t3", q_sigma=2.0, seq_len=150, sel_width=120, hole_frac=0.0, dup_frac=0.3),
])
def test_random_cases_match_dense_masked(oracle_mod, kw):
    w = wl.random_case(seed=hash(str(sorted(kw.items()))) % 10000, **kw)
    _assert_close(oracle_mod.decode_workload(w), dense_masked(w))


def test_row_subset_matches_full(oracle_mod):
    w = wl.random_case(num_seqs=4, heads=2, seq_len=120, sel_width=30, seed=7)
    full = oracle_mod.decode_workload(w)
    part = oracle_mod.decode_workload(w, rows=[3, 1])
    np.testing.assert_array_equal(part, full[[3, 1]])


# ---------------------------------------------------------------------------------
# Closed forms.
# ---------------------------------------------------------------------------------

def _manual_case(cache_rows, sel, seq_len, block_size, heads=1, q=None, k_scale=1.0,
                 v_scale=1.0, sm_scale=1.0):
    """A one-sequence case with the given cache rows (uint8 [n, 512]) laid out in pages."""
    n = cache_rows.shape[0]
    pages = (n + block_size - 1) // block_size
    cache = np.zeros((pages, block_size * 512), dtype=np.uint8)
    cache.reshape(-1)[: n * 512] = cache_rows.reshape(-1)
    bt = np.arange(pages, dtype=np.int32).reshape(1, -1)
    if q is None:
        q = torch.zeros((1, heads, 512), dtype=torch.bfloat16)
    return wl.Workload("manual", q, torch.from_numpy(cache), None, torch.from_numpy(bt),
                       torch.tensor([seq_len], dtype=torch.int32),
                       torch.tensor([sel], dtype=torch.int32), 1, 1, q.shape[1], block_size,
                       block_size * 512, pages, k_scale, v_scale, sm_scale)


def test_two_token_worked_example(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "two_token_worked_example.json")))
    rows = np.zeros((2, 512), dtype=np.uint8)
    rows[0, 0], rows[1, 0] = 0x38, 0x40
    rows[0, 1] = 0x38
    q = torch.zeros((1, 1, 512), dtype=torch.bfloat16)
    q[0, 0, 0] = 1.0
    w = _manual_case(rows, g["selection"], g["seq_len"], g["block_size"], q=q)
    out = oracle_mod.decode_workload(w)[0, 0]
    assert out[0] == pytest.approx(g["expected_dim0"], rel=1e-15)
    assert out[1] == pytest.approx(g["expected_dim1"], rel=1e-15)
    assert np.all(out[2:] == 0.0)


def test_single_token_returns_scaled_row(oracle_mod):
    w = wl.random_case(heads=5, seq_len=300, sel_width=16, hole_frac=0.0, dup_frac=0.0, seed=3)
    sel = w.sel_indices.clone()
    j = int(sel[0, 7])
    sel[0, :] = -1
    sel[0, 3] = j
    sel[0, 11] = j          # a duplicate of the same token changes nothing
    w.sel_indices = sel
    out = oracle_mod.decode_workload(w)
    h = w.host()
    page = int(h["block_tables"][0, j // w.block_size])
    off = page * w.cache_stride_bytes + (j % w.block_size) * 512
    row = _fp8_bytes_to_f64(h["k_cache"].reshape(-1)[off:off + 512])
    for head in range(5):
        np.testing.assert_array_equal(out[0, head], w.v_scale * row)


def test_all_holes_give_zero(oracle_mod):
    w = wl.random_case(num_seqs=2, heads=3, seq_len=64, sel_width=12, seed=4)
    sel = w.sel_indices.clone()
    sel[1] = -1
    sel[1, 0] = 64            # == seq_len: out of range, also a hole
    sel[1, 1] = -7
    w.sel_indices = sel
    out = oracle_mod.decode_workload(w)
    assert np.all(out[1] == 0.0)
    assert np.any(out[0] != 0.0)


def test_zero_query_gives_mean(oracle_mod):
    w = wl.random_case(heads=2, seq_len=128, sel_width=40, seed=5)
    w.q = torch.zeros_like(w.q)
    out = oracle_mod.decode_workload(w)
    h = w.host()
    ids, cnt = oracle_mod.resolve_indices(h["sel_indices"], h["seq_lens"])
    kc = h["k_cache"].reshape(-1)
    rows = []
    for j in ids[0, :cnt[0]]:
        page = int(h["block_tables"][0, j // w.block_size])
        off = page * w.cache_stride_bytes + (j % w.block_size) * 512
        rows.append(_fp8_bytes_to_f64(kc[off:off + 512]))
    mean = w.v_scale * np.mean(rows, axis=0)
    _assert_close(out[0, 0], mean)
    _assert_close(out[0, 1], mean)


def test_dominant_score_selects_argmax(oracle_mod):
    w = wl.random_case(heads=3, seq_len=200, sel_width=30, hole_frac=0.0, dup_frac=0.0, seed=6)
    w.sm_scale = 1e4
    out = oracle_mod.decode_workload(w)
    dm = dense_masked(w)
    _assert_close(out, dm)
    # every head's output equals (up to rounding) one selected row
    h = w.host()
    kc = h["k_cache"].reshape(-1)
    cands = []
    for j in set(int(x) for x in h["sel_indices"][0] if 0 <= x < 200):
        page = int(h["block_tables"][0, j // w.block_size])
        off = page * w.cache_stride_bytes + (j % w.block_size) * 512
        cands.append(w.v_scale * _fp8_bytes_to_f64(kc[off:off + 512]))
    cands = np.stack(cands)
    for head in range(3):
        d = np.abs(cands - out[0, head][None, :]).max(axis=1)
        assert d.min() < 1e-9


# ---------------------------------------------------------------------------------
# Invariants.
# ---------------------------------------------------------------------------------

def test_invariants_permutation_duplicates_holes(oracle_mod):
    w = wl.random_case(num_seqs=2, heads=4, seq_len=180, sel_width=50, seed=8)
    base = oracle_mod.decode_workload(w)
    sel = w.sel_indices.clone()
    g = torch.Generator().manual_seed(9)
    # permute
    w.sel_indices = sel[:, torch.randperm(sel.shape[1], generator=g)].contiguous()
    np.testing.assert_array_equal(oracle_mod.decode_workload(w), base)
    # duplicate every id and append holes / out-of-range ids (wider row)
    extra = torch.tensor([[-1, 180, 10**6, -3]] * 2, dtype=torch.int32)
    w.sel_indices = torch.cat([sel, sel, extra], dim=1).contiguous()
    np.testing.assert_array_equal(oracle_mod.decode_workload(w), base)


# ---------------------------------------------------------------------------------
# Multi-row (verify) semantics.
# ---------------------------------------------------------------------------------

def test_verify_row_lengths_rule(oracle_mod):
    # decode_k.rs decode_k: row r sits at seq_len + r and its seq_len entry is pos + 1.
    got = oracle_mod.verify_row_lengths(np.array([10, 20]), 3)
    np.testing.assert_array_equal(got, [11, 12, 13, 21, 22, 23])


def test_verify_rows_see_only_their_prefix(oracle_mod):
    # k = 3 verify rows of one sequence select the same ids; row r may not see the
    # token written for a later row.
    base, k = 40, 3
    w = wl.random_case(num_seqs=1, rows_per_seq=k, heads=2, seq_lens=[base + r + 1 for r in range(k)],
                       block_size=16, sel_width=20, seed=10)
    sel = w.sel_indices.clone()
    sel[:] = sel[0]
    sel[:, 0] = base + 2          # only visible to the last row
    w.sel_indices = sel
    out = oracle_mod.decode_workload(w)
    _assert_close(out, dense_masked(w))
    assert not np.allclose(out[2], out[0])


def test_bad_page_is_reported(oracle_mod):
    w = wl.random_case(heads=1, seq_len=64, sel_width=8, hole_frac=0.0, dup_frac=0.0, seed=11)
    bt = w.block_tables.clone()
    bt[0, :] = 10**6
    w.block_tables = bt
    with pytest.raises(ValueError):
        oracle_mod.decode_workload(w)

"""The roofline numerator of bench.py (algorithmic bytes and flops of a step), checked on
the CPU against an independent count with Python sets."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from sparse_mla_paged_gb300 import workloads as wl  # noqa: E402


def _count(w):
    sel = w.sel_indices.numpy()
    lens = w.seq_lens.numpy()
    R, W = sel.shape
    rows = [{int(j) for j in sel[r] if 0 <= j < lens[r]} for r in range(R)]
    tokens, pages = 0, 0
    for s in range(w.num_seqs):
        union = set().union(*rows[s * w.rows_per_seq:(s + 1) * w.rows_per_seq])
        tokens += len(union)
        pages += len({j // w.block_size for j in union})
    kv = tokens * 512 * (1 if w.v_cache is None else 2)
    qb = R * w.num_q_heads * 512 * 2
    selected = sum(len(x) for x in rows)
    return kv + 2 * qb + R * W * 4 + pages * 4, 4 * w.num_q_heads * 512 * selected


def test_tiny_cost_by_hand():
    w = wl.tiny()
    c = bench.algorithmic_cost(w)
    # 55 distinct ids (the rest are holes or copies), 4 heads, one row of 64 slots
    assert c["selected_tokens"] == 55 and c["union_tokens"] == 55
    pages = len({int(j) // 64 for j in w.sel_indices.numpy()[0] if 0 <= j < 256})
    assert c["bytes"] == 55 * 512 + 2 * 4 * 512 * 2 + 64 * 4 + pages * 4
    assert c["flops"] == 4 * 4 * 512 * 55


def test_cost_matches_set_count():
    cases = [
        wl.random_case(num_seqs=3, rows_per_seq=2, heads=5, seq_lens=[100, 101, 40, 41, 300, 301], block_size=16,
                       sel_width=64, dup_frac=0.2, out_of_range_frac=0.1, seed=31),
        wl.random_case(num_seqs=2, heads=3, seq_len=500, block_size=32, sel_width=128, split_kv=True, seed=32),
    ]
    for w in cases:
        c = bench.algorithmic_cost(w)
        want_bytes, want_flops = _count(w)
        assert c["bytes"] == want_bytes and c["flops"] == want_flops

"""CPU oracle for the selected-index (DSA) NoPE MLA paged decode.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference arm may import this package. The product path (the
``sparse_mla_paged_gb300`` package and its CUDA library) never imports, links or calls
it, and it shares no code with that path.

The arithmetic lives in ``dsa_oracle.c`` (plain C, IEEE double); this module builds it
with gcc and marshals numpy arrays into it. Each function names the passage of the
source pages it restates:

* ``attend.rs`` = spark_model/layers/glm5next_dsa/attend.rs
* ``decode_k.rs`` = metrale_model_arch/glm5next_dsa/layer/decode_k.rs

* ``build.rs`` = spark_model/layers/glm5next_dsa/build.rs

The cache writer (``latent_write``, ``e4m3_encode``) restates the ``latent_write`` launch
of decode_k.rs ``decode_k``; its kernel body is not on the pages and the reading taken is
written beside ``oracle_latent_write`` in ``dsa_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdsa_oracle.so")
_lock = threading.Lock()
_lib = None

LATENT = 512


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, pthreads). Returns the shared-library path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    """Load an oracle shared library at ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f64.restype = f64
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = f64
    lib.oracle_e4m3_table.argtypes = [P]
    lib.oracle_e4m3_table.restype = None
    lib.oracle_resolve_indices.argtypes = [P, P, i32, i32, P, P]
    lib.oracle_resolve_indices.restype = i32
    lib.oracle_dsa_mla_decode.argtypes = [P, P, P, i64, P, i32, P, P, i32, i32, i32, i32,
                                          i32, i64, f64, f64, f64, P, i32, P, i32]
    lib.oracle_dsa_mla_decode.restype = i32
    lib.oracle_online_cores.argtypes = []
    lib.oracle_online_cores.restype = i32
    lib.oracle_e4m3_encode.argtypes = [f64]
    lib.oracle_e4m3_encode.restype = ctypes.c_uint8
    lib.oracle_latent_write.argtypes = [P, P, P, i32, f64, f64, i32, i64, P, i64, P]
    lib.oracle_latent_write.restype = i32
    lib.oracle_select_pools.argtypes = [P, P, i32, i32, i32, i32, P]
    lib.oracle_select_pools.restype = i32
    for name in ("oracle_absorb_q", "oracle_absorb_o"):
        getattr(lib, name).argtypes = [P, P, i32, i32, i32, i32, i32, i64, i64, P]
        getattr(lib, name).restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
        return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def e4m3_table(lib=None) -> np.ndarray:
    """All 256 E4M3 codes decoded to float64 (OCP FP8 E4M3, the "fn" variant)."""
    out = np.zeros(256, dtype=np.float64)
    (lib or _load()).oracle_e4m3_table(_ptr(out))
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
    return np.array([lib.oracle_bf16_to_f64(int(b)) for b in flat]).reshape(np.shape(bits))


def online_cores() -> int:
    return int(_load().oracle_online_cores())


def resolve_indices(sel_indices: np.ndarray, seq_lens: np.ndarray, lib=None):
    """Per row: the ascending distinct ids with 0 <= id < seq_lens[r], padded with -1.

    attend.rs module doc ("Why this is not the masked kernel"): -1 marks a hole and the
    mask is set membership with duplicates collapsed. Returns (ids [rows, W], counts [rows]).
    """
    sel = np.ascontiguousarray(sel_indices, dtype=np.int32)
    rows, width = sel.shape
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32).reshape(rows)
    ids = np.empty((rows, width), dtype=np.int32)
    counts = np.empty(rows, dtype=np.int32)
    rc = (lib or _load()).oracle_resolve_indices(_ptr(sel), _ptr(lens), width, rows, _ptr(ids),
                                        _ptr(counts))
    if rc != 0:
        raise ValueError("oracle_resolve_indices: bad arguments")
    return ids, counts


def verify_row_lengths(base_lens: np.ndarray, k: int) -> np.ndarray:
    """decode_k.rs ``decode_k``: row ``r`` of a k-row verify pass sits at position
    ``seq_len + r`` and its seq_len entry is ``pos + 1``. Returns [num_seqs * k] lengths."""
    base = np.asarray(base_lens, dtype=np.int64).reshape(-1)
    return (base[:, None] + np.arange(k, dtype=np.int64)[None, :] + 1).reshape(-1).astype(np.int32)


def decode(q_bits, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices,
           num_seqs, rows_per_seq, num_q_heads, block_size, cache_stride_bytes,
           k_scale, v_scale, sm_scale, rows=None, threads: int = 0, lib=None) -> np.ndarray:
    """The decode of attend.rs ``decode_attention`` in float64, for the decode rows in
    ``rows`` (all rows when None). Returns float64 [len(rows), num_q_heads, 512].

    q_bits: uint16 BF16 bit patterns [R, H, 512]; k_cache / v_cache: uint8 E4M3 codes
    (any shape, read as flat bytes); block_tables: int32 [*, max_blocks_per_seq] (row
    stride max_blocks_per_seq, 0 = one shared row); seq_lens: int32 [R] per decode row;
    sel_indices: int32 [R, W].
    """
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kc = np.ascontiguousarray(k_cache, dtype=np.uint8).reshape(-1)
    vc = kc if v_cache is None else np.ascontiguousarray(v_cache, dtype=np.uint8).reshape(-1)
    if vc.size != kc.size:
        raise ValueError("k_cache and v_cache must have the same size")
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32).reshape(-1)
    sel = np.ascontiguousarray(sel_indices, dtype=np.int32)
    total_rows = num_seqs * rows_per_seq
    if rows is None:
        rows = np.arange(total_rows, dtype=np.int32)
    rows = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1)
    if q.shape != (total_rows, num_q_heads, LATENT):
        raise ValueError(f"q shape {q.shape} != {(total_rows, num_q_heads, LATENT)}")
    if sel.shape[0] != total_rows or lens.size != total_rows:
        raise ValueError("sel_indices / seq_lens row count mismatch")
    out = np.zeros((rows.size, num_q_heads, LATENT), dtype=np.float64)
    rc = (lib or _load()).oracle_dsa_mla_decode(
        _ptr(q), _ptr(kc), _ptr(vc), kc.size, _ptr(bt), int(max_blocks_per_seq), _ptr(lens),
        _ptr(sel), sel.shape[1], int(num_seqs), int(rows_per_seq), int(num_q_heads),
        int(block_size), int(cache_stride_bytes), float(k_scale), float(v_scale),
        float(sm_scale), _ptr(rows), rows.size, _ptr(out), int(threads))
    if rc == -2:
        raise ValueError("a selected token resolves outside the cache (bad block table)")
    if rc != 0:
        raise ValueError("oracle_dsa_mla_decode: bad arguments")
    return out


def decode_workload(w, rows=None, threads: int = 0, lib=None) -> np.ndarray:
    """Convenience: run :func:`decode` on a workload object's host copies."""
    h = w.host()
    return decode(h["q_bits"], h["k_cache"], h["v_cache"], h["block_tables"],
                  w.max_blocks_per_seq, h["seq_lens"], h["sel_indices"], w.num_seqs,
                  w.rows_per_seq, w.num_q_heads, w.block_size, w.cache_stride_bytes,
                  w.k_scale, w.v_scale, w.sm_scale, rows=rows, threads=threads, lib=lib)


def e4m3_encode(values, lib=None) -> np.ndarray:
    """E4M3 ("fn") codes of float64 values: round to nearest even, saturating to +-448."""
    lib = lib or _load()
    flat = np.ascontiguousarray(values, dtype=np.float64).ravel()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in flat], dtype=np.uint8).reshape(np.shape(values))


def latent_write(kv_a_bits, weight_bits, slots, rms_eps, kv_scale, block_size, cache_stride_bytes, cache,
                 lib=None):
    """decode_k.rs ``decode_k``, the ``latent_write`` launch: RMSNorm(kv_a) * w * (1/kv_scale)
    stored as E4M3 at each row's slot (negative slot: skipped). ``cache`` (uint8, flat view
    of the pool) is written in place. 1/kv_scale is formed in single precision, as the
    launcher does. Returns the float64 values before rounding, [rows, 512]."""
    x = np.ascontiguousarray(kv_a_bits, dtype=np.uint16).reshape(-1, LATENT)
    w = np.ascontiguousarray(weight_bits, dtype=np.uint16).reshape(LATENT)
    sl = np.ascontiguousarray(slots, dtype=np.int64).reshape(-1)
    if sl.size != x.shape[0]:
        raise ValueError("one slot per row")
    if not (cache.flags["C_CONTIGUOUS"] and cache.dtype == np.uint8):
        raise ValueError("cache must be a contiguous uint8 array")
    inv = float(np.float32(1.0) / np.float32(kv_scale))
    vals = np.zeros((x.shape[0], LATENT), dtype=np.float64)
    rc = (lib or _load()).oracle_latent_write(_ptr(x), _ptr(w), _ptr(sl), x.shape[0], float(rms_eps), inv,
                                              int(block_size), int(cache_stride_bytes), _ptr(cache),
                                              cache.size, _ptr(vals))
    if rc == -2:
        raise ValueError("a slot falls outside the cache")
    if rc != 0:
        raise ValueError("oracle_latent_write: bad arguments")
    return vals


def select_pools(scores, q_pos, kpool: int, topk: int, lib=None) -> np.ndarray:
    """The selector the decode's input comes from (attend.rs module doc; decode_k.rs
    decode_k): per row, the ``topk`` highest-scoring pools among those ending at or before
    q_pos (equal scores: lower pool first; NaN lowest), listed in ascending position as
    ``kpool`` consecutive token ids each, -1 padded to ``topk * kpool``. scores: float32
    [rows, n_pools]; q_pos: int32 [rows]. Returns int32 [rows, topk * kpool]."""
    sc = np.ascontiguousarray(scores, dtype=np.float32)
    rows, n_pools = sc.shape
    qp = np.ascontiguousarray(q_pos, dtype=np.int32).reshape(rows)
    out = np.empty((rows, topk * kpool), dtype=np.int32)
    rc = (lib or _load()).oracle_select_pools(_ptr(sc), _ptr(qp), rows, n_pools, int(kpool), int(topk), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_select_pools: bad arguments")
    return out


def _bf16_bits(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("BF16 inputs are passed as uint16 bit patterns")
    return np.ascontiguousarray(a)


def absorb_q(q_b, kv_b, heads: int, nope: int, vd: int, kvl: int = LATENT, rows=None, lib=None) -> np.ndarray:
    """build.rs ``absorb_q``: q_absorb[h*kvl + c, k] = sum_r kv_b[h*(nope+vd) + r, c] *
    q_b[h*nope + r, k] in float64. q_b: BF16 bits [heads*nope, ql]; kv_b: BF16 bits
    [heads*(nope+vd), kvl]. rows=(row0, nrows) computes only those output rows.
    Returns float64 [nrows, ql]."""
    qb, kb = _bf16_bits(q_b), _bf16_bits(kv_b)
    ql = qb.shape[1]
    if qb.shape != (heads * nope, ql) or kb.shape != (heads * (nope + vd), kvl):
        raise ValueError("absorb_q: shapes do not match heads/nope/vd/kvl")
    row0, nrows = rows if rows is not None else (0, heads * kvl)
    out = np.empty((nrows, ql), dtype=np.float64)
    rc = (lib or _load()).oracle_absorb_q(_ptr(qb), _ptr(kb), heads, nope, vd, kvl, ql, row0, nrows, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_absorb_q: bad arguments")
    return out


def absorb_o(o_proj, kv_b, heads: int, nope: int, vd: int, kvl: int = LATENT, rows=None, lib=None) -> np.ndarray:
    """build.rs ``absorb_o``: o_absorb[i, h*kvl + c] = sum_r o_proj[i, h*vd + r] *
    kv_b[h*(nope+vd) + nope + r, c] in float64 (the V half of kv_b). o_proj: BF16 bits
    [hidden, heads*vd]; kv_b as for absorb_q. rows=(row0, nrows) computes only those
    output rows. Returns float64 [nrows, heads*kvl]."""
    op, kb = _bf16_bits(o_proj), _bf16_bits(kv_b)
    hidden = op.shape[0]
    if op.shape != (hidden, heads * vd) or kb.shape != (heads * (nope + vd), kvl):
        raise ValueError("absorb_o: shapes do not match heads/nope/vd/kvl")
    row0, nrows = rows if rows is not None else (0, hidden)
    out = np.empty((nrows, heads * kvl), dtype=np.float64)
    rc = (lib or _load()).oracle_absorb_o(_ptr(op), _ptr(kb), heads, nope, vd, kvl, hidden, row0, nrows, _ptr(out))
    if rc != 0:
        raise ValueError("oracle_absorb_o: bad arguments")
    return out

"""Python binding of the C ABI (include/dsa_mla.h): argument marshalling only.

Every step of the decode runs in the library's sm_103a kernels; these functions pass
torch tensors' device pointers, sizes and the current CUDA stream through ctypes and
raise DsaError on a non-OK status.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib
from ._lib import DsaError, check  # noqa: F401

LATENT = 512


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: torch.Tensor, dtype, name: str):
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor of {dtype}")


def abi_version() -> int:
    return int(_lib.load().dsa_abi_version())


def status_string(status: int) -> str:
    return _lib.load().dsa_status_string(int(status)).decode()


def _decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices, num_seqs,
                 rows_per_seq, num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale, out):
    _need(q, torch.bfloat16, "q")
    _need(k_cache, torch.uint8, "k_cache")
    _need(v_cache, torch.uint8, "v_cache")
    _need(block_tables, torch.int32, "block_tables")
    _need(seq_lens, torch.int32, "seq_lens")
    _need(sel_indices, torch.int32, "sel_indices")
    _need(out, torch.bfloat16, "out")
    return [_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), int(max_blocks_per_seq), _ptr(seq_lens),
            _ptr(sel_indices), int(sel_indices.shape[-1]), int(num_seqs), int(rows_per_seq), int(num_q_heads),
            int(block_size), int(cache_stride_bytes), float(k_scale), float(v_scale), float(sm_scale), _ptr(out)]


def _out_like(q, out):
    return torch.empty_like(q) if out is None else out


def decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices, num_seqs,
           rows_per_seq, num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale,
           out=None, stream=None) -> torch.Tensor:
    """dsa_mla_decode: per-row seq_lens; returns out (bf16 [R, H, 512])."""
    out = _out_like(q, out)
    a = _decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices, num_seqs,
                     rows_per_seq, num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale, out)
    check(_lib.load().dsa_mla_decode(*a, _stream(stream)), "dsa_mla_decode")
    return out


def decode_k(q, k_cache, v_cache, block_tables, max_blocks_per_seq, base_lens, sel_indices, num_seqs, k,
             num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale, out=None,
             stream=None) -> torch.Tensor:
    """dsa_mla_decode_k: k verify rows per sequence; base_lens is per sequence."""
    out = _out_like(q, out)
    a = _decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, base_lens, sel_indices, num_seqs, k,
                     num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale, out)
    check(_lib.load().dsa_mla_decode_k(*a, _stream(stream)), "dsa_mla_decode_k")
    return out


def workspace_bytes(num_seqs, rows_per_seq, num_q_heads, sel_width, num_ctas=0) -> int:
    return int(_lib.load().dsa_mla_decode_workspace_bytes(int(num_seqs), int(rows_per_seq), int(num_q_heads),
                                                          int(sel_width), int(num_ctas)))


def decode_grid(num_seqs, rows_per_seq, num_q_heads, sel_width, num_ctas=0) -> int:
    """Decode grid size a call of this shape runs with (dsa_mla_decode_grid; 0 = none)."""
    return int(_lib.load().dsa_mla_decode_grid(int(num_seqs), int(rows_per_seq), int(num_q_heads),
                                               int(sel_width), int(num_ctas)))


def alloc_workspace(num_seqs, rows_per_seq, num_q_heads, sel_width, num_ctas=0, device=None) -> torch.Tensor:
    n = workspace_bytes(num_seqs, rows_per_seq, num_q_heads, sel_width, num_ctas)
    if n == 0:
        raise DsaError(2, "dsa_mla_decode_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device or "cuda")


def options(num_ctas=0, tile_tokens=0, wait_limit_ns=0, ev_begin=None, ev_end=None,
            gather_mode=0) -> "_lib.DecodeOptions":
    """A dsa_decode_options struct (zero fields take the library defaults)."""
    o = _lib.DecodeOptions()
    o.num_ctas = int(num_ctas)
    o.tile_tokens = int(tile_tokens)
    o.gather_mode = int(gather_mode)
    o.wait_limit_ns = int(wait_limit_ns)
    o.ev_begin = None if ev_begin is None else ev_begin.cuda_event
    o.ev_end = None if ev_end is None else ev_end.cuda_event
    return o


def decode_ws(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices, num_seqs,
              rows_per_seq, num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale, out,
              workspace: torch.Tensor, verify_rows=0, num_ctas=0, ev_begin=None, ev_end=None,
              tile_tokens=0, wait_limit_ns=0, gather_mode=0, stream=None) -> torch.Tensor:
    """dsa_mla_decode_ws: caller workspace (capturable) and per-call options."""
    a = _decode_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices, num_seqs,
                     rows_per_seq, num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale, out)
    _need(workspace, torch.uint8, "workspace")
    o = options(num_ctas, tile_tokens, wait_limit_ns, ev_begin, ev_end, gather_mode)
    check(_lib.load().dsa_mla_decode_ws(*a, int(verify_rows), _ptr(workspace), workspace.numel(),
                                        _lib.ctypes.byref(o), _stream(stream)), "dsa_mla_decode_ws")
    return out


def host_workspace_bytes(num_seqs, rows_per_seq, num_q_heads, sel_width, table_rows, max_blocks_per_seq,
                         verify_rows=0, num_ctas=0) -> int:
    return int(_lib.load().dsa_mla_decode_host_workspace_bytes(
        int(num_seqs), int(rows_per_seq), int(num_q_heads), int(sel_width), int(table_rows),
        int(max_blocks_per_seq), int(verify_rows), int(num_ctas)))


def decode_host(q_host, k_cache, v_cache, block_tables_host, max_blocks_per_seq, seq_lens_host, sel_host,
                num_seqs, rows_per_seq, num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale,
                out_host, workspace, verify_rows=0, num_ctas=0, stream=None) -> torch.Tensor:
    """dsa_mla_decode_host: per-step inputs and output in (pinned) host memory."""
    for t, n in ((q_host, "q_host"), (block_tables_host, "block_tables_host"), (seq_lens_host, "seq_lens_host"),
                 (sel_host, "sel_host"), (out_host, "out_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    _need(k_cache, torch.uint8, "k_cache")
    _need(v_cache, torch.uint8, "v_cache")
    check(_lib.load().dsa_mla_decode_host(
        _ptr(q_host), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables_host), int(block_tables_host.shape[0]),
        int(max_blocks_per_seq), _ptr(seq_lens_host), _ptr(sel_host), int(sel_host.shape[-1]), int(num_seqs),
        int(rows_per_seq), int(num_q_heads), int(block_size), int(cache_stride_bytes), float(k_scale),
        float(v_scale), float(sm_scale), _ptr(out_host), int(verify_rows), _ptr(workspace), workspace.numel(),
        int(num_ctas), _stream(stream)), "dsa_mla_decode_host")
    return out_host


def resolve_indices(sel_indices: torch.Tensor, seq_lens: torch.Tensor, stream=None):
    """dsa_resolve_indices -> (ids int32 [rows, W], counts int32 [rows])."""
    _need(sel_indices, torch.int32, "sel_indices")
    _need(seq_lens, torch.int32, "seq_lens")
    rows, width = sel_indices.shape
    ids = torch.empty((rows, width), dtype=torch.int32, device=sel_indices.device)
    counts = torch.empty(rows, dtype=torch.int32, device=sel_indices.device)
    check(_lib.load().dsa_resolve_indices(_ptr(sel_indices), _ptr(seq_lens), int(width), int(rows), _ptr(ids),
                                          _ptr(counts), _stream(stream)), "dsa_resolve_indices")
    return ids, counts


def latent_write(kv_a: torch.Tensor, norm_weight: torch.Tensor, slots: torch.Tensor, rms_eps: float,
                 kv_scale: float, block_size: int, cache_stride_bytes: int, cache: torch.Tensor,
                 stream=None) -> torch.Tensor:
    """dsa_latent_write: RMSNorm(kv_a) * weight * (1/kv_scale) as E4M3 into each row's slot of
    the paged cache (negative slot: skipped). Returns cache."""
    _need(kv_a, torch.bfloat16, "kv_a")
    _need(norm_weight, torch.bfloat16, "norm_weight")
    _need(slots, torch.int64, "slots")
    _need(cache, torch.uint8, "cache")
    if kv_a.shape[-1] != LATENT or norm_weight.numel() != LATENT or slots.numel() != kv_a.numel() // LATENT:
        raise ValueError("kv_a [rows, 512], norm_weight [512], slots [rows]")
    check(_lib.load().dsa_latent_write(_ptr(kv_a), _ptr(norm_weight), _ptr(slots), int(slots.numel()),
                                       float(rms_eps), float(kv_scale), int(block_size), int(cache_stride_bytes),
                                       _ptr(cache), _stream(stream)), "dsa_latent_write")
    return cache


def select_pools(scores: torch.Tensor, q_pos: torch.Tensor, kpool: int, topk: int, out=None,
                 stream=None) -> torch.Tensor:
    """dsa_select_pools: per row the topk highest-scoring pools ending at or before q_pos, as
    ascending token ids (kpool per pool), -1 padded; returns int32 [rows, topk * kpool]."""
    _need(scores, torch.float32, "scores")
    _need(q_pos, torch.int32, "q_pos")
    rows, n_pools = scores.shape
    if out is None:
        out = torch.empty((rows, topk * kpool), dtype=torch.int32, device=scores.device)
    _need(out, torch.int32, "out")
    check(_lib.load().dsa_select_pools(_ptr(scores), _ptr(q_pos), int(rows), int(n_pools), int(kpool), int(topk),
                                       _ptr(out), _stream(stream)), "dsa_select_pools")
    return out


def _absorb_out(shape, dtype, device, out):
    if dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("absorb output must be float32 or bfloat16")
    if out is None:
        out = torch.empty(shape, dtype=dtype, device=device)
    _need(out, dtype, "out")
    if tuple(out.shape) != tuple(shape):
        raise ValueError(f"out must have shape {tuple(shape)}")
    return out, 0 if dtype == torch.float32 else 1


def absorb_q(q_b: torch.Tensor, kv_b: torch.Tensor, heads: int, nope: int, vd: int, dtype=torch.float32, out=None,
             stream=None) -> torch.Tensor:
    """dsa_absorb_q (build.rs absorb_q): q_b bf16 [heads*nope, q_lora_rank], kv_b bf16
    [heads*(nope+vd), kvl] -> [heads*kvl, q_lora_rank] in `dtype` (float32 or bfloat16)."""
    _need(q_b, torch.bfloat16, "q_b")
    _need(kv_b, torch.bfloat16, "kv_b")
    ql, kvl = q_b.shape[1], kv_b.shape[1]
    if q_b.shape[0] != heads * nope or kv_b.shape[0] != heads * (nope + vd):
        raise ValueError("absorb_q: shapes do not match heads/nope/vd")
    out, code = _absorb_out((heads * kvl, ql), dtype, q_b.device, out)
    check(_lib.load().dsa_absorb_q(_ptr(q_b), _ptr(kv_b), heads, nope, vd, kvl, ql, _ptr(out), code,
                                   _stream(stream)), "dsa_absorb_q")
    return out


def absorb_o(o_proj: torch.Tensor, kv_b: torch.Tensor, heads: int, nope: int, vd: int, dtype=torch.float32,
             out=None, stream=None) -> torch.Tensor:
    """dsa_absorb_o (build.rs absorb_o): o_proj bf16 [hidden, heads*vd], kv_b bf16
    [heads*(nope+vd), kvl] -> [hidden, heads*kvl] in `dtype` (float32 or bfloat16)."""
    _need(o_proj, torch.bfloat16, "o_proj")
    _need(kv_b, torch.bfloat16, "kv_b")
    hidden, kvl = o_proj.shape[0], kv_b.shape[1]
    if o_proj.shape[1] != heads * vd or kv_b.shape[0] != heads * (nope + vd):
        raise ValueError("absorb_o: shapes do not match heads/nope/vd")
    out, code = _absorb_out((hidden, heads * kvl), dtype, o_proj.device, out)
    check(_lib.load().dsa_absorb_o(_ptr(o_proj), _ptr(kv_b), heads, nope, vd, kvl, hidden, _ptr(out), code,
                                   _stream(stream)), "dsa_absorb_o")
    return out


def read_device_status(workspace: torch.Tensor, stream=None) -> int:
    v = _lib.ctypes.c_int32(0)
    check(_lib.load().dsa_read_device_status(_ptr(workspace), _lib.ctypes.byref(v), _stream(stream)),
          "dsa_read_device_status")
    return int(v.value)


def last_device_status(stream=None) -> int:
    v = _lib.ctypes.c_int32(0)
    check(_lib.load().dsa_last_device_status(_lib.ctypes.byref(v), _stream(stream)), "dsa_last_device_status")
    return int(v.value)


def static_device_status(stream=None) -> int:
    """Device status word of the latest dsa_mla_decode_static call on the current device."""
    v = _lib.ctypes.c_int32(0)
    check(_lib.load().dsa_static_device_status(_lib.ctypes.byref(v), _stream(stream)), "dsa_static_device_status")
    return int(v.value)


# ----------------------------------------------------------------------------------------
# Workload conveniences (a workloads.Workload holds the tensors and the scalars).
# ----------------------------------------------------------------------------------------

def _workload_args(w):
    vc = w.k_cache if w.v_cache is None else w.v_cache
    return (w.q, w.k_cache, vc, w.block_tables, w.max_blocks_per_seq)


def decode_workload(w, out=None, workspace=None, num_ctas=0, verify=None, stream=None, ev_begin=None,
                    ev_end=None, tile_tokens=0, wait_limit_ns=0, gather_mode=0) -> torch.Tensor:
    """Run the decode on a Workload. verify=True uses the k-row entry point with the
    workload's per-sequence base lengths. Per-call options (num_ctas, tile_tokens,
    wait_limit_ns, gather_mode, events) go through dsa_mla_decode_ws; without a workspace one is
    allocated for the call."""
    q, kc, vc, bt, mbps = _workload_args(w)
    out = torch.empty_like(q) if out is None else out
    verify = (w.base_lens is not None) if verify is None else verify
    lens = w.base_lens if verify else w.seq_lens
    if workspace is None and (num_ctas or tile_tokens or wait_limit_ns or gather_mode or ev_begin is not None):
        workspace = alloc_workspace(w.num_seqs, w.rows_per_seq, w.num_q_heads, w.sel_width, num_ctas,
                                    device=q.device)
    if workspace is None:
        fn = decode_k if verify else decode
        return fn(q, kc, vc, bt, mbps, lens, w.sel_indices, w.num_seqs, w.rows_per_seq, w.num_q_heads,
                  w.block_size, w.cache_stride_bytes, w.k_scale, w.v_scale, w.sm_scale, out=out, stream=stream)
    return decode_ws(q, kc, vc, bt, mbps, lens, w.sel_indices, w.num_seqs, w.rows_per_seq, w.num_q_heads,
                     w.block_size, w.cache_stride_bytes, w.k_scale, w.v_scale, w.sm_scale, out, workspace,
                     verify_rows=1 if verify else 0, num_ctas=num_ctas, ev_begin=ev_begin, ev_end=ev_end,
                     tile_tokens=tile_tokens, wait_limit_ns=wait_limit_ns, gather_mode=gather_mode,
                     stream=stream)

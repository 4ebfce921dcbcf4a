"""Helpers shared by the GPU parity tests (no decode arithmetic here)."""
import numpy as np
import torch

from sparse_mla_paged_gb300 import workloads as wl

ATOL = 1e-2
RTOL = 1e-2


def assert_parity(gpu_out: torch.Tensor, ref: np.ndarray, what: str = ""):
    """|gpu - ref| <= 1e-2 + 1e-2*|ref| for every element (gpu BF16, ref float64)."""
    got = gpu_out.detach().float().cpu().numpy().astype(np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any() or not np.isfinite(got).all():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} elements outside |err| <= {ATOL} + {RTOL}|ref|; "
            f"worst at {idx}: gpu {got[idx]:.6g} ref {ref[idx]:.6g}; max err {err.max():.4g}; "
            f"nonfinite {int((~np.isfinite(got)).sum())}")
    return float(err.max())


def sub_workload(w: wl.Workload, seqs) -> wl.Workload:
    """The sequences `seqs` of w (all their rows) with only their pages, on the CPU.

    The touched bytes are identical; pages are re-numbered 0.. in table order. Used so
    that the oracle can evaluate sampled rows of full-size workloads without a host copy
    of the whole pool."""
    seqs = list(seqs)
    rps = w.rows_per_seq
    rows = [s * rps + i for s in seqs for i in range(rps)]
    bt = w.block_tables
    mbps = bt.shape[1]
    shared = w.max_blocks_per_seq == 0
    tables = bt[[0] if shared else seqs].to(torch.int64)             # [S', mbps]
    cache = w.k_cache.reshape(w.k_cache.shape[0], -1)
    pages = tables.reshape(-1)
    valid = pages >= 0
    src = torch.where(valid, pages, torch.zeros_like(pages))
    kc = cache[src.to(cache.device)].cpu()
    vc = None if w.v_cache is None else w.v_cache.reshape(cache.shape[0], -1)[src.to(cache.device)].cpu()
    new_bt = torch.arange(pages.numel(), dtype=torch.int32).reshape(tables.shape)
    new_bt[~valid.cpu().reshape(tables.shape)] = -1
    sub = wl.Workload(w.name + f" [seqs {seqs}]", w.q[rows].cpu(), kc, vc, new_bt, w.seq_lens[rows].cpu(),
                      w.sel_indices[rows].cpu(), len(seqs), rps, w.num_q_heads, w.block_size,
                      w.cache_stride_bytes, 0 if shared else mbps, w.k_scale, w.v_scale, w.sm_scale,
                      None if w.base_lens is None else w.base_lens[seqs].cpu())
    return sub, rows

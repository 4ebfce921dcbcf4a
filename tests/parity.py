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


def sub_workload(w: wl.Workload, seqs):
    """The sequences `seqs` of w with only their pages, on the CPU (see Workload.subset)."""
    return w.subset(seqs)

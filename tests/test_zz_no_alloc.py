"""The allocation-free entry point, dsa_mla_decode_static.

It serves callers that cannot allocate device memory when they call the decode (code
under a framework that owns all device memory, or latency-critical paths that cannot take
cudaMalloc's synchronisation) and keep no workspace of their own: its scratch is a fixed
device array inside the library. These checks call it through the C ABI and compare it
with dsa_mla_decode (the library-workspace entry point) and with the CPU oracle on two
different calls in a row, element by element within the parity tolerance
(|err| <= 1e-2 + 1e-2*|ref|); check that its device status word is readable without any
allocation (a bad block-table entry reports DSA_ERR_DEVICE_BOUNDS, the next clean call
DSA_OK); and check that a shape too large for the array is refused before anything runs.

This file is collected last, so that a run that stops at the first failure has run every
other test first; it also passes on its own in a fresh process.
"""
import pytest
import torch

import oracle
from parity import assert_parity
from sparse_mla_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


@pytest.fixture(scope="module")
def libs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_paged_gb300 import build
    build.build()
    import sparse_mla_paged_gb300.api as api
    lib = api._lib.load()
    torch.cuda.set_device(0)
    return api, lib


def _static_call(lib, w, out, stream):
    vc = w.k_cache if w.v_cache is None else w.v_cache
    return lib.dsa_mla_decode_static(
        w.q.data_ptr(), w.k_cache.data_ptr(), vc.data_ptr(), w.block_tables.data_ptr(), w.max_blocks_per_seq,
        w.seq_lens.data_ptr(), w.sel_indices.data_ptr(), w.sel_width, w.num_seqs, w.rows_per_seq,
        w.num_q_heads, w.block_size, w.cache_stride_bytes, w.k_scale, w.v_scale, w.sm_scale, out.data_ptr(),
        stream)


def test_static_matches_library_workspace_two_calls(libs):
    api, lib = libs
    stream = torch.cuda.current_stream().cuda_stream
    cases = [
        wl.random_case(num_seqs=2, heads=64, seq_lens=[4096, 3000], sel_width=2048, hole_frac=0.02,
                       dup_frac=0.0, seed=4141),
        wl.random_case(num_seqs=3, heads=96, seq_lens=[700, 2300, 90], sel_width=900, hole_frac=0.05,
                       dup_frac=0.05, out_of_range_frac=0.02, seed=4242),
    ]
    for w_cpu in cases:                  # two calls in a row, different shapes
        w = w_cpu.to("cuda")
        want = api.decode_workload(w)    # dsa_mla_decode
        got = torch.empty_like(w.q)
        assert _static_call(lib, w, got, stream) == 0
        torch.cuda.synchronize()
        assert api.static_device_status() == 0
        g, r = got.float(), want.float()
        assert torch.isfinite(g).all()
        err = (g - r).abs()
        assert bool((err <= ATOL + RTOL * r.abs()).all()), f"max err {err.max().item():.4g}"
        assert_parity(got, oracle.decode_workload(w_cpu), f"static entry point vs oracle, {w_cpu.name}")


def test_static_device_status_reports_a_bad_page(libs):
    api, lib = libs
    stream = torch.cuda.current_stream().cuda_stream
    w = wl.random_case(num_seqs=2, heads=8, seq_len=300, sel_width=100, hole_frac=0.0, dup_frac=0.0, seed=13)
    bt = w.block_tables.clone()
    bt[1, 2] = -5                        # a negative page for sequence 1 ...
    sel = w.sel_indices.clone()
    sel[1, 0] = 2 * 64 + 3               # ... that the selection uses
    w.block_tables, w.sel_indices = bt, sel
    wd = w.to("cuda")
    out = torch.empty_like(wd.q)
    assert _static_call(lib, wd, out, stream) == 0
    assert api.static_device_status() == 6           # DSA_ERR_DEVICE_BOUNDS
    w.block_tables = w.block_tables.abs()
    wd = w.to("cuda")
    assert _static_call(lib, wd, out, stream) == 0
    assert api.static_device_status() == 0


def test_static_rejects_oversize_shape(libs):
    api, lib = libs
    w = wl.random_case(heads=8, seq_len=300, sel_width=100, device="cuda", seed=7)
    # the same buffers, described as 4096 rows x 128 heads x 8192 selected: far beyond the
    # array, so the call must return DSA_ERR_WORKSPACE without enqueuing anything
    n = api.workspace_bytes(4096, 1, 128, 8192)
    assert n > 40 * 1024 * 1024
    rc = lib.dsa_mla_decode_static(
        w.q.data_ptr(), w.k_cache.data_ptr(), w.k_cache.data_ptr(), w.block_tables.data_ptr(),
        w.max_blocks_per_seq, w.seq_lens.data_ptr(), w.sel_indices.data_ptr(), 8192, 4096, 1, 128, w.block_size,
        w.cache_stride_bytes, w.k_scale, w.v_scale, w.sm_scale, w.q.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert rc == 3
    torch.cuda.synchronize()

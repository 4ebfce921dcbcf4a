"""GPU parity of the cache writer (dsa_latent_write, decode_k.rs decode_k: the latent_write
launch) against the CPU oracle, and a decode of rows it wrote.

The stored codes must equal the oracle's, except where the oracle's float64 value before
rounding lies within a relative 2^-17 of a rounding midpoint of E4M3: there the kernel's
single-precision norm (a reduction and rsqrtf, a few units of 2^-23) may fall on either
side, and either neighbouring code is correct. Bytes outside the written rows must not
change.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity
from sparse_mla_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
L = 512
TIE = 2.0 ** -17


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_mla_paged_gb300 import build
    build.build()
    import sparse_mla_paged_gb300.api as api
    api._lib.load()
    torch.cuda.set_device(0)
    return api


def _inputs(rows, bs, pages, seed, x_scale=1.0):
    g = np.random.default_rng(seed)
    x = torch.from_numpy((g.normal(size=(rows, L)) * x_scale).astype(np.float32)).to(torch.bfloat16)
    w = torch.from_numpy(g.uniform(0.5, 1.5, L).astype(np.float32)).to(torch.bfloat16)
    slots = g.permutation(pages * bs)[:rows].astype(np.int64)
    if rows > 2:
        slots[rows // 2] = -1                                  # a row that writes nothing
    return x, w, slots


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16)


def assert_written(gpu: np.ndarray, ora: np.ndarray, vals: np.ndarray, slots, bs, stride, what=""):
    written = np.zeros(gpu.size, dtype=bool)
    for r, slot in enumerate(slots):
        if slot < 0:
            continue
        base = (slot // bs) * stride + (slot % bs) * L
        written[base:base + L] = True
        g, o = gpu[base:base + L], ora[base:base + L]
        bad = np.nonzero(g != o)[0]
        if bad.size:
            v = vals[r, bad]
            lo = oracle.e4m3_encode(v * (1 - TIE))
            hi = oracle.e4m3_encode(v * (1 + TIE))
            ok = (lo != hi) & ((g[bad] == lo) | (g[bad] == hi))
            assert ok.all(), (f"{what}: row {r} dims {bad[~ok][:8]}: gpu {g[bad][~ok][:8]} oracle "
                              f"{o[bad][~ok][:8]} values {v[~ok][:8]}")
    assert np.array_equal(gpu[~written], ora[~written]), f"{what}: bytes outside the written rows changed"


@pytest.mark.parametrize("rows,bs,pad,kv_scale,x_scale", [
    (1, 64, 0, 0.05, 1.0), (37, 64, 0, 0.05, 3.0), (200, 16, 80, 0.005, 1.0), (64, 1, 0, 0.05, 0.01),
    (50, 100, 0, 0.1, 20.0), (300, 64, 0, 0.02, 1.0)])
def test_writer_parity(api, rows, bs, pad, kv_scale, x_scale):
    pages = max(4, (rows + bs - 1) // bs + 3)
    stride = bs * L + pad
    x, w, slots = _inputs(rows, bs, pages, seed=rows * 7 + bs, x_scale=x_scale)
    start = np.random.default_rng(rows).integers(0, 256, pages * stride, dtype=np.uint8)
    ora = start.copy()
    vals = oracle.latent_write(_bits(x), _bits(w), slots, 1e-6, kv_scale, bs, stride, ora)
    cache = torch.from_numpy(start.copy()).cuda()
    api.latent_write(x.cuda(), w.cuda(), torch.from_numpy(slots).cuda(), 1e-6, kv_scale, bs, stride, cache)
    torch.cuda.synchronize()
    assert_written(cache.cpu().numpy(), ora, vals, slots, bs, stride, f"rows {rows} bs {bs}")
    if kv_scale == 0.005:                                      # values past 448 saturate
        assert (np.abs(vals) > 448).any()


def test_zero_rows_and_zero_vector(api):
    cache = torch.zeros(4 * 64 * L, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, L), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(L, dtype=torch.bfloat16, device="cuda")
    cache.fill_(7)
    api.latent_write(x[:0], w, torch.zeros(0, dtype=torch.int64, device="cuda"), 1e-6, 0.05, 64, 64 * L, cache)
    api.latent_write(x, w, torch.tensor([70], dtype=torch.int64, device="cuda"), 1e-6, 0.05, 64, 64 * L, cache)
    torch.cuda.synchronize()
    c = cache.cpu().numpy()
    assert np.all(c[70 * L:71 * L] == 0) and np.all(np.delete(c, np.s_[70 * L:71 * L]) == 7)


def test_written_rows_decode(api):
    """The last ten positions of two sequences are rewritten by the writer and selected by
    their rows; the decode of the written cache matches the oracle's write-then-decode."""
    w = wl.random_case(num_seqs=2, heads=64, seq_len=700, sel_width=300, seed=31)
    bs = w.block_size
    bt = w.block_tables.numpy()
    pos = np.arange(690, 700)
    slots = np.array([bt[s, p // bs] * bs + p % bs for s in range(2) for p in pos], dtype=np.int64)
    x, wt, _ = _inputs(len(slots), bs, 4, seed=5, x_scale=2.0)
    sel = w.sel_indices.clone()
    sel[:, :10] = torch.from_numpy(pos.astype(np.int32))
    w.sel_indices = sel
    # oracle: write into a host copy of the pool, then decode it
    ora_cache = w.k_cache.numpy().copy()
    oracle.latent_write(_bits(x), _bits(wt), slots, 1e-6, w.k_scale, bs, w.cache_stride_bytes, ora_cache.reshape(-1))
    w_ora = wl.Workload(**{**w.__dict__, "k_cache": torch.from_numpy(ora_cache), "_host": None})
    ref = oracle.decode_workload(w_ora)
    # GPU: write into the device pool, then decode it
    wd = w.to("cuda")
    api.latent_write(x.cuda(), wt.cuda(), torch.from_numpy(slots).cuda(), 1e-6, w.k_scale, bs, w.cache_stride_bytes,
                     wd.k_cache)
    out = api.decode_workload(wd)
    torch.cuda.synchronize()
    assert_parity(out, ref, "decode of rows written by dsa_latent_write")


def test_writer_rejects_bad_arguments(api):
    x = torch.zeros((2, L), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(L, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(2, dtype=torch.int64, device="cuda")
    cache = torch.zeros(64 * L, dtype=torch.uint8, device="cuda")
    for kw in (dict(kv_scale=0.0), dict(rms_eps=-1.0), dict(block_size=0), dict(stride=64 * L - 16)):
        with pytest.raises(api.DsaError) as e:
            api.latent_write(x, w, s, kw.get("rms_eps", 1e-6), kw.get("kv_scale", 0.05), kw.get("block_size", 64),
                             kw.get("stride", 64 * L), cache)
        assert e.value.status == 1

"""GPU parity: the sm_103a decode through the C ABI against the CPU oracle.

Bar: index resolution bit-exact; every BF16 output element within
|err| <= 1e-2 + 1e-2*|ref| of the float64 oracle.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity, sub_workload
from sparse_mla_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


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


def _run(api, w, **kw):
    wd = w.to("cuda")
    out = api.decode_workload(wd, **kw)
    torch.cuda.synchronize()
    return out


def _check(api, w, what="", status_ok=True, **kw):
    ref = oracle.decode_workload(w)
    if "workspace" in kw and kw["workspace"] is None:
        kw.pop("workspace")
    out = _run(api, w, **kw)
    err = assert_parity(out, ref, what or w.name)
    if status_ok:
        assert api.last_device_status() == 0
    return out, err


# ------------------------------------------------------------------------------------
# Index resolution: bit-exact.
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("rows,width,maxlen", [(1, 1, 1), (7, 64, 300), (40, 2048, 5000), (9, 513, 70000),
                                               (6, 8192, 8500), (5, 2048, 262144), (3, 4096, 300000),
                                               (4, 8192, 2_000_000), (3, 2048, 5_000_000)])
def test_resolve_bit_exact(api, rows, width, maxlen):
    g = np.random.default_rng(rows * 1000 + width)
    sel = g.integers(-3, maxlen + 50, size=(rows, width)).astype(np.int32)
    sel[g.random((rows, width)) < 0.1] = -1
    if width > 4:
        sel[:, width // 2:width // 2 + 3] = sel[:, :3]              # duplicates
    lens = g.integers(0, maxlen + 1, size=rows).astype(np.int32)
    lens[0] = maxlen
    if rows > 1:
        sel[1] = -1                                                 # all holes
    ids, cnt = api.resolve_indices(torch.from_numpy(sel).cuda(), torch.from_numpy(lens).cuda())
    torch.cuda.synchronize()
    rid, rcnt = oracle.resolve_indices(sel, lens)
    np.testing.assert_array_equal(cnt.cpu().numpy(), rcnt)
    np.testing.assert_array_equal(ids.cpu().numpy(), rid)


# ------------------------------------------------------------------------------------
# Decode parity on small cases that span several tiles and ragged tails.
# ------------------------------------------------------------------------------------

def test_tiny_config(api):
    _check(api, wl.tiny())


CASES = {
    "one tile": dict(heads=4, seq_len=256, sel_width=64),
    "ragged 3 tiles": dict(heads=64, seq_len=1000, sel_width=300, hole_frac=0.05),
    "many tiles": dict(heads=64, seq_len=5000, sel_width=2048, hole_frac=0.02, dup_frac=0.0),
    "two head groups": dict(heads=128, seq_len=900, sel_width=500),
    "96 heads": dict(heads=96, seq_len=700, sel_width=260, out_of_range_frac=0.05),
    "130 heads": dict(heads=130, seq_len=400, sel_width=129),
    "one head": dict(heads=1, seq_len=300, sel_width=200),
    "block size 1": dict(heads=16, seq_len=200, block_size=1, sel_width=150),
    "block size 100": dict(heads=16, seq_len=1234, block_size=100, sel_width=400),
    "block size 16": dict(heads=32, seq_len=3000, block_size=16, sel_width=1000),
    "padded stride": dict(heads=8, seq_len=500, block_size=32, sel_width=200, stride_pad=80),
    "split K/V": dict(heads=64, seq_len=800, sel_width=400, split_kv=True),
    "split K/V many tiles": dict(heads=8, seq_len=3000, sel_width=1500, split_kv=True),
    "shared table": dict(num_seqs=3, heads=8, seq_len=600, sel_width=200, shared_table=True),
    "multi seq": dict(num_seqs=6, heads=64, seq_lens=[300, 1000, 40, 5000, 129, 2048], sel_width=700),
    "rows per seq": dict(num_seqs=3, rows_per_seq=2, heads=16, seq_lens=[500, 501, 90, 91, 2000, 2001],
                         sel_width=400),
    "width 1": dict(heads=4, seq_len=100, sel_width=1, hole_frac=0.0, dup_frac=0.0),
    "heavy tails": dict(heads=64, seq_len=3000, sel_width=1024, cache_dist="t3", q_sigma=2.0),
    "peaky scores": dict(heads=16, seq_len=1000, sel_width=512, q_sigma=4.0, cache_dist="t3"),
    "scales": dict(heads=8, seq_len=600, sel_width=300, k_scale=0.3, v_scale=0.01, sm_scale=0.2),
    "negative score scale": dict(heads=8, seq_len=600, sel_width=300, sm_scale=-0.05),
}


@pytest.mark.parametrize("name", list(CASES))
def test_decode_cases(api, name):
    _check(api, wl.random_case(seed=zlib.crc32(name.encode()) % 100000, **CASES[name]), name)


@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("name", ["ragged 3 tiles", "many tiles", "130 heads", "block size 1", "split K/V many tiles",
                                  "multi seq", "rows per seq", "heavy tails", "negative score scale"])
def test_decode_cases_forced_tile(api, name, tile):
    """Both builds of the decode kernel (64- and 128-token tiles) on the same inputs."""
    w = wl.random_case(seed=zlib.crc32(name.encode()) % 100000, **CASES[name])
    _check(api, w, f"{name} tile {tile}", tile_tokens=tile, status_ok=False)


@pytest.mark.parametrize("ctas", [1, 2, 3, 5, 17, 64, 152, 400])
def test_decode_cta_counts(api, ctas):
    w = wl.random_case(num_seqs=4, heads=96, seq_lens=[2000, 100, 1500, 3000], sel_width=1000, seed=77)
    ws = api.alloc_workspace(w.num_seqs, w.rows_per_seq, w.num_q_heads, w.sel_width, num_ctas=ctas)
    _check(api, w, f"{ctas} CTAs", workspace=ws, num_ctas=ctas, status_ok=False)
    assert api.read_device_status(ws) == 0


def _aligned_default(units, slots, sms):
    c_max = max(1, min(sms, -(-slots // 128)))
    for c in range(c_max, 0, -1):
        if 4 * c < 3 * c_max:
            break
        if c % units == 0 or units % c == 0:
            return c
    return c_max


@pytest.mark.parametrize("seqs,k,heads,width", [(128, 1, 128, 2048), (64, 1, 64, 2048), (32, 4, 64, 2048),
                                                 (8, 1, 64, 2048), (80, 1, 64, 2048), (1, 1, 4, 64),
                                                 (3, 1, 64, 300)])
def test_default_grid_prefers_unit_alignment(api, seqs, k, heads, width):
    """The default grid: at most one CTA per SM and 128 slots per CTA, and the largest
    count that is a multiple or a divisor of the unit count when it is at least 3/4 of
    that bound (no CTA then changes unit in mid-range)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = seqs * k * ((heads + 63) // 64)
    got = api.decode_grid(seqs, k, heads, width)
    assert got == _aligned_default(units, units * width, sms)
    if sms == 152 and (seqs, k, heads) in ((128, 1, 128), (64, 1, 64), (32, 4, 64), (8, 1, 64)):
        assert got == 128                    # the four large workloads' shapes on GB300
    assert api.decode_grid(seqs, k, heads, width, 5) == 5


def test_default_grid_sizes_the_default_workspace(api):
    """The workspace sized for the default grid equals the one sized for the grid that
    dsa_mla_decode_grid reports."""
    for seqs, k, heads, width in [(128, 1, 128, 2048), (64, 1, 64, 2048), (3, 1, 64, 300), (80, 1, 64, 2048)]:
        c = api.decode_grid(seqs, k, heads, width)
        assert c > 0
        assert api.workspace_bytes(seqs, k, heads, width) == api.workspace_bytes(seqs, k, heads, width, c)


def test_default_grid_decodes_whole_units_without_combine(api):
    """Eight rows of 64 heads on 4 CTAs (two whole units each): parity, and every CTA
    boundary on a unit boundary."""
    w = wl.random_case(num_seqs=8, heads=64, seq_len=900, sel_width=256, seed=21)
    ws = api.alloc_workspace(8, 1, 64, 256, num_ctas=4)
    _check(api, w, "4 CTAs over 8 units", workspace=ws, num_ctas=4, status_ok=False)
    assert api.read_device_status(ws) == 0


@pytest.mark.parametrize("width,ctas", [(10, 15), (64, 100)])
def test_more_ctas_than_slots(api, width, ctas):
    """CTAs without slots leave no piece; the combine skips them."""
    w = wl.random_case(heads=64, seq_len=300, sel_width=width, hole_frac=0.0, dup_frac=0.0, seed=width)
    ws = api.alloc_workspace(1, 1, 64, width, num_ctas=ctas)
    _check(api, w, f"{ctas} CTAs over {width} slots", workspace=ws, num_ctas=ctas, status_ok=False)
    assert api.read_device_status(ws) == 0


def test_empty_and_single_token_rows(api):
    w = wl.random_case(num_seqs=4, heads=64, seq_len=700, sel_width=300, hole_frac=0.0, dup_frac=0.0, seed=5)
    sel = w.sel_indices.clone()
    sel[1] = -1                            # all holes
    sel[2] = -1
    sel[2, 17] = 650                       # one token
    sel[2, 200] = 650                      # ... duplicated
    sel[3, :] = 700 + torch.arange(300)    # every id out of range
    w.sel_indices = sel
    for ctas in (0, 9):
        ws = None if ctas == 0 else api.alloc_workspace(4, 1, 64, 300, num_ctas=ctas)
        out, _ = _check(api, w, f"empty rows ctas={ctas}", workspace=ws, num_ctas=ctas)
        o = out.float().cpu()
        assert torch.all(o[1] == 0) and torch.all(o[3] == 0)
    # single token: v_scale * V of that token, to BF16 rounding
    h = w.host()
    page = int(h["block_tables"][2, 650 // 64])
    off = page * w.cache_stride_bytes + (650 % 64) * 512
    row = torch.from_numpy(h["k_cache"].reshape(-1)[off:off + 512].copy()).view(torch.float8_e4m3fn).float()
    want = (row * w.v_scale).to(torch.bfloat16).float()
    assert torch.equal(o[2], want.expand_as(o[2]))


def test_invariants_on_gpu(api):
    w = wl.random_case(num_seqs=2, heads=64, seq_len=3000, sel_width=1000, seed=8)
    base = _run(api, w).cpu()
    g = torch.Generator().manual_seed(1)
    perm = w.sel_indices[:, torch.randperm(w.sel_width, generator=g)].contiguous()
    w2 = wl.Workload(**{**w.__dict__, "sel_indices": perm, "_host": None})
    assert torch.equal(_run(api, w2).cpu(), base)               # same set, same partition: bit-identical
    wider = torch.cat([w.sel_indices, w.sel_indices[:, :300], torch.full((2, 50), -1, dtype=torch.int32)], 1)
    w3 = wl.Workload(**{**w.__dict__, "sel_indices": wider.contiguous(), "_host": None})
    out3 = _run(api, w3).cpu()
    assert_parity(out3, oracle.decode_workload(w), "duplicates + holes")


def test_zero_query_gives_mean(api):
    w = wl.random_case(heads=64, seq_len=2000, sel_width=700, seed=9)
    w.q = torch.zeros_like(w.q)
    _check(api, w, "zero query")


# ------------------------------------------------------------------------------------
# Multi-row (verify) entry point.
# ------------------------------------------------------------------------------------

def test_decode_k_matches_per_row_semantics(api):
    k, S = 3, 4
    base = [500, 1200, 64, 3000]
    lens = oracle.verify_row_lengths(np.array(base), k)
    w = wl.random_case(num_seqs=S, rows_per_seq=k, heads=64, seq_lens=lens.tolist(), sel_width=600, seed=10)
    sel = w.sel_indices.clone()
    for s in range(S):
        for r in range(k):
            sel[s * k + r, 0] = base[s] + k - 1        # the last row's new token: visible to it only
    w.sel_indices = sel
    w.base_lens = torch.tensor(base, dtype=torch.int32)
    ref = oracle.decode_workload(w)
    out = _run(api, w, verify=True)
    assert_parity(out, ref, "decode_k")
    out_rows = _run(api, w, verify=False)                # per-row lengths through dsa_mla_decode
    assert torch.equal(out.cpu(), out_rows.cpu())


# ------------------------------------------------------------------------------------
# Host-buffer entry point, graph capture, device status.
# ------------------------------------------------------------------------------------

def test_decode_host_matches_device(api):
    w = wl.random_case(num_seqs=3, heads=64, seq_lens=[900, 2500, 100], sel_width=800, seed=11)
    wd = w.to("cuda")
    dev = api.decode_workload(wd)
    n = api.host_workspace_bytes(w.num_seqs, 1, w.num_q_heads, w.sel_width, w.block_tables.shape[0],
                                 w.max_blocks_per_seq)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out_h = torch.empty(w.q.shape, dtype=torch.bfloat16).pin_memory()
    api.decode_host(w.q.pin_memory(), wd.k_cache, wd.k_cache, w.block_tables.pin_memory(), w.max_blocks_per_seq,
                    w.seq_lens.pin_memory(), w.sel_indices.pin_memory(), w.num_seqs, 1, w.num_q_heads,
                    w.block_size, w.cache_stride_bytes, w.k_scale, w.v_scale, w.sm_scale, out_h, ws)
    torch.cuda.synchronize()
    assert torch.equal(out_h, dev.cpu())


def test_graph_capture_replay(api):
    w = wl.random_case(num_seqs=2, heads=128, seq_len=1500, sel_width=900, seed=12).to("cuda")
    ws = api.alloc_workspace(2, 1, 128, 900)
    out = torch.empty_like(w.q)
    api.decode_workload(w, out=out, workspace=ws)
    torch.cuda.synchronize()
    want = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            api.decode_workload(w, out=out, workspace=ws, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, want)


def test_events_around_decode_kernel_outside_capture(api):
    """The optional events bracket the decode kernel on the call's stream, captured or not."""
    w = wl.random_case(num_seqs=2, heads=64, seq_len=3000, sel_width=1024, seed=15).to("cuda")
    ws = api.alloc_workspace(2, 1, 64, 1024)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    e1.record(s)                                   # creates both CUDA events
    want = api.decode_workload(w, workspace=ws)
    got = api.decode_workload(w, workspace=ws, ev_begin=e0, ev_end=e1)
    torch.cuda.synchronize()
    assert torch.equal(got, want)
    assert e0.query() and e1.query()
    assert e0.elapsed_time(e1) >= 0.0


def test_bad_page_sets_device_status(api):
    w = wl.random_case(num_seqs=2, heads=8, seq_len=300, sel_width=100, hole_frac=0.0, dup_frac=0.0, seed=13)
    bt = w.block_tables.clone()
    bt[1, 2] = -5                                  # a negative page for sequence 1
    w.block_tables = bt
    sel = w.sel_indices.clone()
    sel[1, 0] = 2 * 64 + 3                         # make sure the bad page is selected
    w.sel_indices = sel
    wd = w.to("cuda")
    ws = api.alloc_workspace(2, 1, 8, 100)
    api.decode_workload(wd, workspace=ws)
    assert api.read_device_status(ws) == 6         # DSA_ERR_DEVICE_BOUNDS
    # a clean call on the same workspace reports OK again
    w.block_tables = w.block_tables.abs()
    api.decode_workload(w.to("cuda"), workspace=ws)
    assert api.read_device_status(ws) == 0


def test_block_table_overrun_sets_device_status(api):
    w = wl.random_case(heads=8, seq_len=300, sel_width=100, seed=14)
    w.seq_lens = torch.tensor([300 + 64 * 3], dtype=torch.int32)   # longer than the table covers
    sel = w.sel_indices.clone()
    sel[0, 0] = 300 + 64 * 2
    w.sel_indices = sel
    ws = api.alloc_workspace(1, 1, 8, 100)
    api.decode_workload(w.to("cuda"), workspace=ws)
    assert api.read_device_status(ws) == 6


def test_invalid_arguments_on_device(api):
    w = wl.random_case(heads=8, seq_len=300, sel_width=100, seed=15).to("cuda")
    with pytest.raises(api.DsaError) as e:
        api.decode(w.q, w.k_cache, w.k_cache, w.block_tables, w.max_blocks_per_seq, w.seq_lens, w.sel_indices,
                   1, 1, 8, 64, 64 * 512 - 16, 0.05, 0.05, 0.04)
    assert e.value.status == 1
    small = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(api.DsaError) as e:
        api.decode_workload(w, workspace=small)
    assert e.value.status == 3


# ------------------------------------------------------------------------------------
# Full-size workloads, in the launch configuration the benchmark times, on sampled
# sequences the oracle evaluates.
# ------------------------------------------------------------------------------------

FULL = {1: [0, 3, 7], 2: [0, 31, 63], 3: [0, 127], 4: [0, 15, 31]}


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_configs_sampled(api, cfg):
    w = wl.config(cfg, device="cuda")
    out = api.decode_workload(w)
    torch.cuda.synchronize()
    assert api.last_device_status() == 0
    sub, rows = sub_workload(w, FULL[cfg])
    ref = oracle.decode_workload(sub)
    assert_parity(out[rows], ref, f"config {cfg} sampled sequences {FULL[cfg]}")
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------------------------------
# Flat tails: one dominant token and width - 1 tokens with identical scores far below it.
# The probability operand has a finite exponent range; each decode tile must keep the
# tail's weight whatever the gap (4 to 24 log2 units over the heads), wherever the
# dominant token sits (first, middle, last) and however the row is split across CTAs.
# ------------------------------------------------------------------------------------

_FLAT = {}


def _flat(tail_value):
    if tail_value not in _FLAT:
        w = wl.flat_tail(tail_value=tail_value)
        _FLAT[tail_value] = (w, oracle.decode_workload(w))
    return _FLAT[tail_value]


@pytest.mark.parametrize("tail_value", [20.0, 80.0])
@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("ctas", [0, 1, 3, 7])
def test_flat_tail(api, tail_value, tile, ctas):
    w, ref = _flat(tail_value)
    out = _run(api, w, tile_tokens=tile, num_ctas=ctas)
    assert_parity(out, ref, f"flat tail |v| {tail_value * w.v_scale} tile {tile} ctas {ctas}")


# ------------------------------------------------------------------------------------
# The bounded-wait path: a 1 ns wait limit makes the pipeline give up; the call records
# DSA_ERR_TIMEOUT, drains and exits, and the next call on the same workspace is clean.
# ------------------------------------------------------------------------------------

def test_wait_timeout_sets_device_status_and_recovers(api):
    w = wl.random_case(num_seqs=2, heads=64, seq_len=3000, sel_width=1024, seed=21)
    wc = w.to("cuda")
    ws = api.alloc_workspace(2, 1, 64, 1024)
    api.decode_workload(wc, workspace=ws, wait_limit_ns=1)
    torch.cuda.synchronize()
    assert api.read_device_status(ws) == 7         # DSA_ERR_TIMEOUT
    out = api.decode_workload(wc, workspace=ws)
    torch.cuda.synchronize()
    assert api.read_device_status(ws) == 0
    assert_parity(out, oracle.decode_workload(w), "after a timed-out call")


# ------------------------------------------------------------------------------------
# The two gather paths (tensor-map gathers, per-thread copies) fill the same operand
# layout, so the decode gives bit-identical outputs through either.
# ------------------------------------------------------------------------------------

@pytest.mark.parametrize("tile", [64, 128])
@pytest.mark.parametrize("name", ["ragged 3 tiles", "many tiles", "130 heads", "block size 1", "block size 100",
                                  "split K/V many tiles", "multi seq", "rows per seq", "heavy tails"])
def test_gather_paths_agree(api, name, tile):
    w = wl.random_case(seed=zlib.crc32(name.encode()) % 100000, **CASES[name]).to("cuda")
    a = api.decode_workload(w, tile_tokens=tile, gather_mode=2)
    b = api.decode_workload(w, tile_tokens=tile, gather_mode=1)
    torch.cuda.synchronize()
    assert torch.equal(a, b)

"""GPU parity of the selector (dsa_select_pools; attend.rs module doc: the decode's input
rows of token ids with -1 holes; decode_k.rs decode_k: index_topk pools per row, only
pools ending at or before q_pos[r]) against the CPU oracle. Index output: bit-exact.

Cases: rows full of ties, NaN and infinities; subnormals and signed zeros; every row
length relative to index_topk (none eligible, fewer than topk, exactly topk, more); the
pooled 128K shape (128 rows x 32768 pools, 512 of 4) and a mixed-position batch; a row
too long for the shared-memory staging; unaligned rows; then the selector's rows fed to
the decode, against the oracle's select-then-decode.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import assert_parity
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


def _run(api, scores, q_pos, kpool, topk):
    out = api.select_pools(torch.from_numpy(scores).cuda(), torch.from_numpy(q_pos).cuda(), kpool, topk)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _check(api, scores, q_pos, kpool, topk, what):
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    q_pos = np.ascontiguousarray(q_pos, dtype=np.int32)
    got = _run(api, scores, q_pos, kpool, topk)
    want = oracle.select_pools(scores, q_pos, kpool, topk)
    bad = np.nonzero((got != want).any(axis=1))[0]
    assert bad.size == 0, f"{what}: rows {bad[:8]} differ; first: gpu {got[bad[0]][:16]} oracle {want[bad[0]][:16]}"


def _tied(seed, rows, n_pools):
    g = np.random.default_rng(seed)
    s = g.integers(-4, 5, size=(rows, n_pools)).astype(np.float32) * 0.5
    s[g.random((rows, n_pools)) < 0.05] = np.nan
    s[g.random((rows, n_pools)) < 0.02] = np.inf
    s[g.random((rows, n_pools)) < 0.02] = -np.inf
    return s


@pytest.mark.parametrize("kpool,topk,n_pools", [(4, 16, 200), (1, 7, 1000), (8, 300, 700), (4, 1, 5000),
                                                (2, 50, 4099), (4, 512, 32768)])
def test_ties_nan_inf(api, kpool, topk, n_pools):
    rows = 12
    s = _tied(kpool * 100 + topk, rows, n_pools)
    g = np.random.default_rng(topk)
    q = g.integers(-3, n_pools * kpool + 5, size=rows).astype(np.int32)
    q[0] = n_pools * kpool - 1
    q[1] = topk * kpool - 1                       # exactly topk eligible
    q[2] = topk * kpool - 2                       # one fewer
    q[3] = topk * kpool + kpool - 1               # one more
    q[4] = kpool - 2                              # none eligible
    q[5] = -1
    _check(api, s, q, kpool, topk, f"ties kpool {kpool} topk {topk}")


def test_special_values(api):
    n = 3000
    g = np.random.default_rng(3)
    rows = []
    rows.append(np.zeros(n, np.float32))                                        # all equal: lowest pools
    r = np.zeros(n, np.float32); r[::2] = -0.0; rows.append(r)                 # signed zeros are equal
    rows.append(np.full(n, np.nan, np.float32))                                 # all NaN
    sub = (g.integers(1, 1 << 23, size=n).astype(np.uint32)).view(np.float32)  # positive subnormals
    rows.append(sub.copy())
    rows.append(-sub)
    m = g.normal(size=n).astype(np.float32); m[g.random(n) < 0.3] = np.float32(1e-40); rows.append(m)
    rows.append(np.where(g.random(n) < 0.5, np.float32(-np.inf), np.float32(np.inf)).astype(np.float32))
    rows.append(np.full(n, np.finfo(np.float32).max, np.float32))
    s = np.stack(rows)
    q = np.full(len(rows), n * 4 - 1, np.int32)
    for topk in (1, 100, 1499, 2999):
        _check(api, s, q, 4, topk, f"special values topk {topk}")


def test_pooled_128k_shape(api):
    scores, q = wl.pool_scores()
    _check(api, scores.numpy(), q.numpy(), 4, 512, "pooled 128K: 128 rows x 32768 pools, 512 of 4")


def test_mixed_positions(api):
    g = np.random.default_rng(11)
    q = g.integers(0, 131072, size=128).astype(np.int32)
    q[:4] = [0, 2047, 2051, 131071]
    scores, q = wl.pool_scores(q_pos=q, seed=5)
    _check(api, scores.numpy(), q.numpy(), 4, 512, "pooled 128K, positions across the context")


def test_unstaged_long_rows(api):
    scores, q = wl.pool_scores(rows=6, n_pools=50001, kpool=4, seed=9)
    s = scores.numpy()
    s[1, ::3] = 0.25                                                     # a heavy tie at the threshold
    q = q.numpy(); q[2] = 77777; q[3] = 4 * 600 - 1
    _check(api, s, q, 4, 512, "rows longer than the staged limit")


def test_crowded_threshold_bin(api):
    """Rows whose threshold bin (the key's top 11 bits) holds more pools than the staged
    kernel's candidate list: every score in [2, 2.5) (one bin), a constant row with a few
    larger scores, a row of equal scores, and the staged limit itself (40960 pools, two
    rounds of 32768) against one past it."""
    g = np.random.default_rng(21)
    for n in (40960, 40961, 30000):
        s = np.empty((5, n), np.float32)
        s[4] = 1.0                                                      # every pool equal
        s[0] = g.uniform(2.0, 2.5, n)
        s[1] = 0.5
        s[1, g.choice(n, 100, replace=False)] = g.uniform(1, 2, 100)
        s[2] = np.float32(2.25) + g.integers(0, 8, n).astype(np.float32) * np.float32(2.0 ** -20)
        s[3] = g.normal(size=n)
        q = np.full(5, n * 4 - 1, np.int32)
        for topk in (512, 4000, 32767):
            _check(api, s, q, 4, topk, f"crowded threshold bin, {n} pools, topk {topk}")


def test_unaligned_rows(api):
    scores, q = wl.pool_scores(rows=7, n_pools=4097, kpool=2, seed=12)
    _check(api, scores.numpy(), q.numpy(), 2, 1000, "odd pool count (rows start off 16 bytes)")
    rows, n = 7, 4096
    flat = scores.numpy().ravel()
    sub = flat[1:1 + rows * n].reshape(rows, n)                         # base 4 bytes past a 16-byte boundary
    view = torch.from_numpy(flat).cuda()[1:1 + rows * n].view(rows, n)
    assert view.data_ptr() % 16 == 4
    out = api.select_pools(view, torch.from_numpy(q.numpy()).cuda(), 2, 1000)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), oracle.select_pools(sub, q.numpy(), 2, 1000))


def test_empty_inputs(api):
    q = torch.zeros(0, dtype=torch.int32, device="cuda")
    out = api.select_pools(torch.zeros((0, 10), device="cuda"), q, 4, 8)
    assert out.shape == (0, 32)
    out = api.select_pools(torch.zeros((3, 0), device="cuda"), torch.tensor([5, 100, -1], dtype=torch.int32,
                                                                            device="cuda"), 4, 8)
    assert torch.all(out == -1)


def test_selected_rows_decode(api):
    """The selector's rows go straight into the decode: the GPU select-then-decode matches
    the oracle's select-then-decode."""
    w = wl.random_case(num_seqs=3, heads=64, seq_len=1200, sel_width=64 * 4, seed=17)
    kpool, topk = 4, 64
    q_pos = (w.seq_lens.numpy() - 1).astype(np.int32)
    q_pos[1] = 500                                                        # a row that sees less
    scores, q = wl.pool_scores(rows=w.rows, n_pools=1200 // kpool, kpool=kpool, q_pos=q_pos, seed=4)
    w.sel_indices = torch.from_numpy(oracle.select_pools(scores.numpy(), q.numpy(), kpool, topk))
    ref = oracle.decode_workload(w)
    wd = w.to("cuda")
    wd.sel_indices = api.select_pools(scores.cuda(), q.cuda(), kpool, topk)
    out = api.decode_workload(wd)
    torch.cuda.synchronize()
    assert_parity(out, ref, "decode of rows chosen by dsa_select_pools")


def test_select_rejects_bad_arguments(api):
    s = torch.zeros((2, 10), device="cuda")
    q = torch.zeros(2, dtype=torch.int32, device="cuda")
    for kpool, topk in ((0, 4), (4, 0)):
        with pytest.raises(api.DsaError) as e:
            api.select_pools(s, q, kpool, topk)
        assert e.value.status == 1

"""GPU parity of the load-time absorb transforms (dsa_absorb_q, dsa_absorb_o; build.rs
absorb_q and absorb_o) against the CPU oracle, and the absorbed-equals-unabsorbed
identity through the GPU decode.

Bound per element: the GEMM accumulates BF16 products exactly in FP32, so its error is at
most K * 2^-24 * sum_r |a_r b_r| (K = nope or vd terms); the test allows 2^-14 of that
sum (64x the bound). The sum of magnitudes is itself an oracle call, on the absolute
weights. BF16 output adds half a BF16 unit of the value (at most 2^-8 of it, at the bottom
of a binade).
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_mla_paged_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
ABS_TOL = 2.0 ** -14


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


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def abs_bits(t: torch.Tensor) -> np.ndarray:
    return bits(t) & np.uint16(0x7FFF)


def check(got: torch.Tensor, ref: np.ndarray, mag: np.ndarray, what: str):
    g = got.float().cpu().numpy().astype(np.float64)
    tol = ABS_TOL * mag + 1e-30
    if got.dtype == torch.bfloat16:
        tol = tol + 2.0 ** -8 * np.abs(ref)   # half a BF16 unit: up to 2^-8 of the value
    bad = np.abs(g - ref) > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} elements off; worst "
                           f"{np.max(np.abs(g - ref) / tol):.3g}x the bound")


@pytest.mark.parametrize("heads,nope,vd,kvl,ql,hidden", [(4, 64, 96, 512, 384, 200), (2, 256, 256, 512, 100, 33),
                                                         (3, 8, 24, 40, 16, 5)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_absorb_parity(api, heads, nope, vd, kvl, ql, hidden, dtype):
    q_b, kv_b, o_proj = wl.absorb_weights(heads, nope, vd, kvl, ql, hidden, seed=heads * 31 + nope)
    qa = api.absorb_q(q_b.cuda(), kv_b.cuda(), heads, nope, vd, dtype=dtype)
    oa = api.absorb_o(o_proj.cuda(), kv_b.cuda(), heads, nope, vd, dtype=dtype)
    torch.cuda.synchronize()
    check(qa, oracle.absorb_q(bits(q_b), bits(kv_b), heads, nope, vd, kvl),
          oracle.absorb_q(abs_bits(q_b), abs_bits(kv_b), heads, nope, vd, kvl), "absorb_q")
    check(oa, oracle.absorb_o(bits(o_proj), bits(kv_b), heads, nope, vd, kvl),
          oracle.absorb_o(abs_bits(o_proj), abs_bits(kv_b), heads, nope, vd, kvl), "absorb_o")


def test_absorb_model_size_sampled_rows(api):
    """64 heads, nope = vd = 256, kvl 512, q_lora_rank 2048, hidden 6144 (FP32 out):
    sampled output rows against the oracle (which computes rows one by one)."""
    H, nope, vd, kvl, ql, hidden = 64, 256, 256, 512, 2048, 6144
    q_b, kv_b, o_proj = wl.absorb_weights(H, nope, vd, kvl, ql, hidden, device="cuda", seed=5)
    qa = api.absorb_q(q_b, kv_b, H, nope, vd)
    oa = api.absorb_o(o_proj, kv_b, H, nope, vd)
    torch.cuda.synchronize()
    qb, kb, ob = bits(q_b), bits(kv_b), bits(o_proj)
    qba, kba, oba = qb & np.uint16(0x7FFF), kb & np.uint16(0x7FFF), ob & np.uint16(0x7FFF)
    g = np.random.default_rng(0)
    for row in list(g.choice(H * kvl, 6, replace=False)) + [0, H * kvl - 1]:
        ref = oracle.absorb_q(qb, kb, H, nope, vd, kvl, rows=(int(row), 1))
        mag = oracle.absorb_q(qba, kba, H, nope, vd, kvl, rows=(int(row), 1))
        check(qa[int(row):int(row) + 1], ref, mag, f"absorb_q row {row}")
    for row in [0, 3071, hidden - 1]:
        ref = oracle.absorb_o(ob, kb, H, nope, vd, kvl, rows=(row, 1))
        mag = oracle.absorb_o(oba, kba, H, nope, vd, kvl, rows=(row, 1))
        check(oa[row:row + 1], ref, mag, f"absorb_o row {row}")


def test_absorbed_decode_equals_unabsorbed_attention(api):
    """absorb_q on the query input, the GPU decode over an E4M3 cache, absorb_o on its
    latent output: the result matches per-head MLA computed the unabsorbed way (float64,
    over the same dequantised cache rows) within the decode's tolerance, carried through
    the output projection as a relative norm (2e-2)."""
    H, nope, vd, kvl, ql, hidden = 16, 128, 128, 512, 256, 96
    AMP = 4.0  # query gain: scores with a spread of a few units (both sides use it)
    q_b, kv_b, o_proj = wl.absorb_weights(H, nope, vd, kvl, ql, hidden, seed=8)
    w = wl.random_case(num_seqs=2, heads=H, seq_len=600, sel_width=256, hole_frac=0.05, seed=9)
    g = np.random.default_rng(3)
    x = g.normal(size=(w.rows, ql))
    qa = api.absorb_q(q_b.cuda(), kv_b.cuda(), H, nope, vd)
    oa = api.absorb_o(o_proj.cuda(), kv_b.cuda(), H, nope, vd)
    xq = torch.from_numpy(x).float().cuda()
    # per-token query projection into latent space (test scaffolding: the projection is
    # outside the decode), then the BF16 queries the decode takes
    q_lat = torch.einsum("hck,rk->rhc", qa.view(H, kvl, ql), xq) * AMP
    wd = w.to("cuda")
    wd.q = q_lat.to(torch.bfloat16).contiguous()
    o_lat = api.decode_workload(wd)
    out = (o_lat.float().reshape(w.rows, H * kvl) @ oa.T).cpu().numpy().astype(np.float64)
    torch.cuda.synchronize()
    # float64 unabsorbed reference over the same cache rows
    table = oracle.e4m3_table()
    h = w.host()
    Wq = torch.from_numpy(bits(q_b).view(np.int16)).view(torch.bfloat16).double().numpy()
    Wkv = torch.from_numpy(bits(kv_b).view(np.int16)).view(torch.bfloat16).double().numpy()
    Wo = torch.from_numpy(bits(o_proj).view(np.int16)).view(torch.bfloat16).double().numpy()
    ids, counts = oracle.resolve_indices(h["sel_indices"], h["seq_lens"])
    for r in range(w.rows):
        seq = r // w.rows_per_seq
        toks = ids[r, :counts[r]]
        pages = h["block_tables"][seq * (w.max_blocks_per_seq and 1), toks // w.block_size]
        rows = h["k_cache"].reshape(-1)[(pages[:, None].astype(np.int64) * w.cache_stride_bytes
                                         + (toks % w.block_size)[:, None] * kvl + np.arange(kvl)[None, :])]
        C = table[rows] * w.k_scale                                         # dequantised latents
        heads = []
        for hh in range(H):
            qn = Wq[hh * nope:(hh + 1) * nope] @ x[r]
            blk = Wkv[hh * (nope + vd):(hh + 1) * (nope + vd)]
            s = w.sm_scale * AMP * ((C @ blk[:nope].T) @ qn)
            p = np.exp(s - s.max())
            heads.append((p / p.sum()) @ (C @ blk[nope:].T))
        ref = Wo @ np.concatenate(heads)
        err = np.linalg.norm(out[r] - ref) / np.linalg.norm(ref)
        assert err < 2e-2, f"row {r}: relative error {err:.3g}"


def test_absorb_rejects_bad_arguments(api):
    q_b, kv_b, o_proj = wl.absorb_weights(2, 8, 8, 16, 12, 4, device="cuda", seed=1)
    with pytest.raises(ValueError):
        api.absorb_q(q_b, kv_b, 3, 8, 8)
    with pytest.raises(ValueError):
        api.absorb_o(o_proj, kv_b, 2, 8, 8, dtype=torch.float16)

"""Pins of the oracle's load-time transforms (build.rs: absorb_q, absorb_o).

The transforms have a plain definition (two contractions of BF16 weights); what pins them
to something other than themselves is the identity they exist for: attention computed
the unabsorbed way (per-head query, key and value projections of the cached latents, a
softmax, the output projection of the concatenated heads; written here in numpy) equals
attention in the latent space with q_absorb applied to the query input and o_absorb to
the latent output. The scores pin absorb_q alone (the K half of kv_b), the output pins
absorb_o (the V half). Invariants add: a head's weights move only that head's block; the
V half of kv_b does not reach absorb_q nor the K half absorb_o; output-row slices equal
the full result. Planted mistakes in a copy of the oracle must fail them.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")


def bf16(x) -> np.ndarray:
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def val(bits) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def weights(seed, H, nope, vd, kvl, ql, hidden):
    g = np.random.default_rng(seed)
    return (bf16(g.normal(size=(H * nope, ql)) / np.sqrt(ql)), bf16(g.normal(size=(H * (nope + vd), kvl)) / np.sqrt(kvl)),
            bf16(g.normal(size=(hidden, H * vd)) / np.sqrt(H * vd)))


def unabsorbed(x, C, q_b, kv_b, o_proj, H, nope, vd, sm):
    """Per-head MLA written out: q = Wq_h x, k_j = W_UK_h c_j, v_j = W_UV_h c_j."""
    Wq, Wkv, Wo = val(q_b), val(kv_b), val(o_proj)
    heads, scores = [], []
    for h in range(H):
        q = Wq[h * nope:(h + 1) * nope] @ x
        blk = Wkv[h * (nope + vd):(h + 1) * (nope + vd)]
        k = C @ blk[:nope].T
        v = C @ blk[nope:].T
        s = sm * (k @ q)
        p = np.exp(s - s.max())
        heads.append((p / p.sum()) @ v)
        scores.append(s)
    return Wo @ np.concatenate(heads), np.stack(scores)


def absorbed(x, C, q_b, kv_b, o_proj, H, nope, vd, sm, lib):
    kvl = C.shape[1]
    qa = oracle.absorb_q(q_b, kv_b, H, nope, vd, kvl, lib=lib)
    oa = oracle.absorb_o(o_proj, kv_b, H, nope, vd, kvl, lib=lib)
    lat, scores = [], []
    for h in range(H):
        s = sm * (C @ (qa[h * kvl:(h + 1) * kvl] @ x))
        p = np.exp(s - s.max())
        lat.append((p / p.sum()) @ C)
        scores.append(s)
    return oa @ np.concatenate(lat), np.stack(scores)


def _identity_checks(lib) -> bool:
    ok = True
    for seed, (H, nope, vd, kvl, ql, hidden, N) in enumerate([(2, 8, 12, 16, 24, 10, 30), (3, 16, 16, 32, 20, 7, 50),
                                                               (1, 5, 3, 9, 11, 4, 17)]):
        q_b, kv_b, o_proj = weights(seed, H, nope, vd, kvl, ql, hidden)
        g = np.random.default_rng(100 + seed)
        x, C = g.normal(size=ql), g.normal(size=(N, kvl))
        sm = 1.0 / np.sqrt(nope)
        ref, s_ref = unabsorbed(x, C, q_b, kv_b, o_proj, H, nope, vd, sm)
        got, s_got = absorbed(x, C, q_b, kv_b, o_proj, H, nope, vd, sm, lib)
        ok = ok and np.allclose(s_got, s_ref, rtol=1e-11, atol=1e-12) and np.allclose(got, ref, rtol=1e-10, atol=1e-12)
    return bool(ok)


def _invariant_checks(lib) -> bool:
    H, nope, vd, kvl, ql, hidden = 3, 6, 5, 8, 7, 4
    q_b, kv_b, o_proj = weights(7, H, nope, vd, kvl, ql, hidden)
    qa = oracle.absorb_q(q_b, kv_b, H, nope, vd, kvl, lib=lib)
    oa = oracle.absorb_o(o_proj, kv_b, H, nope, vd, kvl, lib=lib)
    ok = True
    # head 1's q_b rows move only rows kvl..2kvl of absorb_q
    q2 = q_b.copy(); q2[nope:2 * nope] = bf16(np.full((nope, ql), 0.5))
    d = np.abs(oracle.absorb_q(q2, kv_b, H, nope, vd, kvl, lib=lib) - qa).sum(axis=1)
    ok = ok and d[kvl:2 * kvl].min() > 0 and d[:kvl].max() == 0 and d[2 * kvl:].max() == 0
    # the V half of kv_b does not reach absorb_q; the K half does not reach absorb_o
    kv_v, kv_k = kv_b.copy(), kv_b.copy()
    for h in range(H):
        kv_v[h * (nope + vd) + nope:(h + 1) * (nope + vd)] = bf16(np.full((vd, kvl), 2.0))
        kv_k[h * (nope + vd):h * (nope + vd) + nope] = bf16(np.full((nope, kvl), -1.0))
    ok = ok and np.array_equal(oracle.absorb_q(q_b, kv_v, H, nope, vd, kvl, lib=lib), qa)
    ok = ok and np.array_equal(oracle.absorb_o(o_proj, kv_k, H, nope, vd, kvl, lib=lib), oa)
    ok = ok and not np.array_equal(oracle.absorb_o(o_proj, kv_v, H, nope, vd, kvl, lib=lib), oa)
    # head 2's o_proj columns move only columns 2kvl..3kvl of absorb_o
    o2 = o_proj.copy(); o2[:, 2 * vd:3 * vd] = bf16(np.full((hidden, vd), 0.25))
    d = np.abs(oracle.absorb_o(o2, kv_b, H, nope, vd, kvl, lib=lib) - oa).sum(axis=0)
    ok = ok and d[2 * kvl:].min() > 0 and d[:2 * kvl].max() == 0
    # output-row slices
    ok = ok and np.array_equal(oracle.absorb_q(q_b, kv_b, H, nope, vd, kvl, rows=(5, 9), lib=lib), qa[5:14])
    ok = ok and np.array_equal(oracle.absorb_o(o_proj, kv_b, H, nope, vd, kvl, rows=(1, 2), lib=lib), oa[1:3])
    return bool(ok)


def test_absorbed_attention_equals_unabsorbed():
    assert _identity_checks(None)


def test_head_locality_halves_and_slices():
    assert _invariant_checks(None)


def test_rejects_mismatched_shapes():
    q_b, kv_b, o_proj = weights(1, 2, 4, 4, 8, 6, 3)
    with pytest.raises(ValueError):
        oracle.absorb_q(q_b, kv_b, 2, 4, 5, 8)
    with pytest.raises(ValueError):
        oracle.absorb_o(o_proj, kv_b, 3, 4, 4, 8)


MUTANTS = {
    "absorb_q reads the V half": ("oracle_bf16_to_f64(kv_b[(h * (nope + vd) + r) * kvl + c]) *",
                                  "oracle_bf16_to_f64(kv_b[(h * (nope + vd) + vd + r) * kvl + c]) *"),
    "absorb_o reads the K half": ("kv_b[(h * (nope + vd) + nope + r) * kvl + c]", "kv_b[(h * (nope + vd) + r) * kvl + c]"),
    "absorb_q uses head 0 of q_b": ("q_b[(h * nope + r) * ql + k]", "q_b[r * ql + k]"),
    "absorb_o uses head 0 of o_proj": ("o_proj[i * in_w + h * vd + r]", "o_proj[i * in_w + r]"),
    "absorb_q drops a term": ("for (int64_t r = 0; r < nope; ++r)", "for (int64_t r = 0; r + 1 < nope; ++r)"),
    "absorb_o drops a term": ("for (int64_t r = 0; r < vd; ++r)", "for (int64_t r = 0; r + 1 < vd; ++r)"),
    "absorb_o output block of head 0": ("out[(i - row0) * out_w + h * kvl + c] = sum;", "out[(i - row0) * out_w + c] = sum;"),
}


def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, old
    path = tmp_path / "m.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libm.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so), str(path), "-lm"])
    return oracle._bind(str(so))


def test_unmutated_copy_passes(tmp_path):
    lib = _build_mutant(tmp_path, "#define LATENT 512", "#define LATENT 512")
    assert _identity_checks(lib) and _invariant_checks(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_absorb_mutant_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, *MUTANTS[name])
    assert not (_identity_checks(lib) and _invariant_checks(lib)), f"planted mistake {name!r} passed every pin"

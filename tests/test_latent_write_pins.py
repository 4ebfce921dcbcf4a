"""Pins of the oracle's cache writer (decode_k.rs, decode_k: the latent_write launch).

The writer's reading is the plain RMSNorm followed by the cache scale and an E4M3 code
(round to nearest even, saturating to +-448) at the slot the decode reads. These checks
tie it to things other than itself:
* the E4M3 encoder against torch's float8_e4m3fn conversion (a library routine) on every
  rounding midpoint of the format and values just around them, and against the format's
  definition for saturation; encode(decode(c)) == c for every finite code (the decoder is
  pinned to torch and the OCP table elsewhere);
* RMSNorm closed forms: a constant vector normalises to +-1 (to 1/2 for x = 1 and
  eps = 3, eps being inside the root), a one-hot vector to
  +-sqrt(512) at its position and 0 elsewhere, the zero vector to 0; scaling the input
  leaves the output unchanged (eps = 0); the weight and 1/kv_scale multiply the output;
* the slot address: only the 512 bytes at (slot / bs)*stride + (slot % bs)*512 change,
  and a negative slot writes nothing.
Planted mistakes in a copy of the oracle must each fail one of them.
"""
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "dsa_oracle.c")
L = 512


def _bf16(x) -> np.ndarray:
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _torch_e4m3(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _finite_values() -> np.ndarray:
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    return np.unique(vals[np.isfinite(vals)])


def _encoder_checks(lib) -> bool:
    vals = _finite_values()                          # ascending, -448 .. 448
    mids = (vals[1:] + vals[:-1]) / 2
    around = np.concatenate([mids, mids * (1 + 2.0 ** -20), mids * (1 - 2.0 ** -20), vals,
                             np.random.default_rng(0).uniform(-448, 448, 4000)])
    around = around[np.abs(around) <= 448]
    # float32 holds every midpoint exactly (a 4-bit significand plus one bit)
    ok = np.array_equal(oracle.e4m3_encode(around, lib=lib), _torch_e4m3(around))
    ok = ok and np.all(oracle.e4m3_encode(np.array([448.0, 449.0, 464.0, 470.0, 479.9, 1e6]), lib=lib) == 0x7E)
    ok = ok and np.all(oracle.e4m3_encode(np.array([-448.5, -1e9]), lib=lib) == 0xFE)
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ok = ok and np.array_equal(oracle.e4m3_encode(dec, lib=lib), codes)
    return bool(ok)


def _write(lib, x, w, slots, eps=1e-6, kv_scale=1.0, bs=4, stride=None, pages=4):
    stride = stride or bs * L
    cache = np.full(pages * stride, 0x5A, dtype=np.uint8)
    vals = oracle.latent_write(_bf16(x), _bf16(w), np.asarray(slots, np.int64), eps, kv_scale, bs, stride, cache,
                               lib=lib)
    return cache, vals


def _norm_checks(lib) -> bool:
    ones = np.ones(L)
    ok = True
    # constant vector: x / rms(x) = sign(x)
    _, v = _write(lib, np.full((1, L), -3.0), ones, [0], eps=0.0)
    ok = ok and np.allclose(v, -1.0, rtol=1e-12)
    # one-hot: sqrt(512) at the position, 0 elsewhere
    x = np.zeros((1, L)); x[0, 17] = 5.0
    _, v = _write(lib, x, ones, [0], eps=0.0)
    ok = ok and abs(v[0, 17] - np.sqrt(L)) < 1e-9 and np.count_nonzero(v) == 1
    # eps inside the root: x = 1 everywhere, eps = 3 gives 1 / sqrt(1 + 3) = 1/2
    _, v = _write(lib, np.ones((1, L)), ones, [0], eps=3.0)
    ok = ok and np.allclose(v, 0.5, rtol=1e-12)
    # zero vector with eps > 0: zeros, not NaN
    _, v = _write(lib, np.zeros((1, L)), ones, [0], eps=1e-5)
    ok = ok and np.all(v == 0.0)
    # scale invariance (eps = 0) and linearity in the weight and in 1/kv_scale
    rng = np.random.default_rng(1)
    x = torch.tensor(rng.normal(size=(2, L)), dtype=torch.float32).to(torch.bfloat16).float().numpy()
    w = torch.tensor(rng.uniform(0.5, 1.5, L), dtype=torch.float32).to(torch.bfloat16).float().numpy()
    _, v1 = _write(lib, x, w, [0, 1], eps=0.0)
    _, v2 = _write(lib, 4.0 * x, w, [0, 1], eps=0.0)
    _, v3 = _write(lib, x, 2.0 * w, [0, 1], eps=0.0)
    _, v4 = _write(lib, x, w, [0, 1], eps=0.0, kv_scale=0.25)
    ok = ok and np.allclose(v1, v2, rtol=1e-12) and np.allclose(v3, 2 * v1, rtol=1e-12)
    ok = ok and np.allclose(v4, 4 * v1, rtol=1e-12)
    # unit weight, eps = 0: mean of squares of the output is 1
    _, v = _write(lib, x, ones, [0, 1], eps=0.0)
    ok = ok and np.allclose((v ** 2).mean(axis=1), 1.0, rtol=1e-12)
    # the stored bytes are the codes of the returned values
    cache, v = _write(lib, x * 40, w, [0, 5], eps=1e-6, kv_scale=0.05, bs=4, stride=4 * L)
    ok = ok and np.array_equal(cache[:L], oracle.e4m3_encode(v[0], lib=lib))
    ok = ok and np.array_equal(cache[1 * 4 * L + 1 * L: 1 * 4 * L + 2 * L], oracle.e4m3_encode(v[1], lib=lib))
    return bool(ok)


def _slot_checks(lib) -> bool:
    rng = np.random.default_rng(2)
    x = rng.normal(size=(3, L)) * 8
    bs, stride = 4, 4 * L + 80                     # padded page stride
    cache, _ = _write(lib, x, np.ones(L), [6, -1, 13], bs=bs, stride=stride, pages=5)
    touched = np.nonzero(cache != 0x5A)[0]
    want = set(range(1 * stride + 2 * L, 1 * stride + 3 * L)) | set(range(3 * stride + 1 * L, 3 * stride + 2 * L))
    return set(touched.tolist()) <= want and len(touched) > L  # some codes may equal 0x5A by chance


def _all_pins(lib) -> bool:
    return _encoder_checks(lib) and _norm_checks(lib) and _slot_checks(lib)


def test_encoder_matches_torch_and_the_format():
    assert _encoder_checks(None)


def test_rmsnorm_closed_forms():
    assert _norm_checks(None)


def test_slot_addressing():
    assert _slot_checks(None)


MUTANTS = {
    "ties away from zero": ("double m = nearbyint(ldexp(a, 9));", "double m = round(ldexp(a, 9));"),
    "normal ties away": ("double m = nearbyint((2.0 * f - 1.0) * 8.0);", "double m = round((2.0 * f - 1.0) * 8.0);"),
    "bias 8": ("(uint8_t)((e + 7) << 3)", "(uint8_t)((e + 8) << 3)"),
    "no saturation": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 480.0) return sign | 0x7E;"),
    "sum instead of mean": ("sqrt(sumsq / LATENT + rms_eps)", "sqrt(sumsq + rms_eps)"),
    "eps outside the root": ("1.0 / sqrt(sumsq / LATENT + rms_eps)", "1.0 / (sqrt(sumsq / LATENT) + rms_eps)"),
    "weight dropped": ("* inv_rms * oracle_bf16_to_f64(weight[c]) * inv_kv_scale", "* inv_rms * inv_kv_scale"),
    "scale dropped": ("* oracle_bf16_to_f64(weight[c]) * inv_kv_scale;", "* oracle_bf16_to_f64(weight[c]);"),
    "slot page from slot % bs": ("(slot / block_size) * cache_stride_bytes", "(slot % block_size) * cache_stride_bytes"),
    "negative slot written": ("if (slot < 0) continue;", "if (slot < -1) continue;"),
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
    assert _all_pins(_build_mutant(tmp_path, "#define LATENT 512", "#define LATENT 512"))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_writer_mutant_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, *MUTANTS[name])
    try:
        passed = _all_pins(lib)
    except ValueError:
        passed = False
    assert not passed, f"planted mistake {name!r} passed every pin"

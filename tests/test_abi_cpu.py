"""C ABI checks that need no GPU: the library loads, exports every entry point the
header declares with the signatures the binding uses, and rejects invalid arguments on
the host before touching CUDA."""
import ctypes
import re

import pytest

from sparse_mla_paged_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    from sparse_mla_paged_gb300 import build
    build.build()
    return _lib.load()


def _declared_functions():
    text = open(_lib.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_\w+)\s*\(", text)))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for want in ("dsa_mla_decode", "dsa_mla_decode_k", "dsa_mla_decode_ws", "dsa_resolve_indices",
                 "dsa_mla_decode_workspace_bytes", "dsa_mla_decode_grid", "dsa_status_string", "dsa_read_device_status",
                 "dsa_mla_decode_host", "dsa_latent_write", "dsa_select_pools", "dsa_absorb_q", "dsa_absorb_o"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no binding signature"


def test_status_strings(lib):
    assert lib.dsa_abi_version() == 2
    for code, name in _lib.STATUS.items():
        s = lib.dsa_status_string(code).decode()
        assert s and s != "unknown status", name
    assert lib.dsa_status_string(99).decode() == "unknown status"


# A valid-looking argument set with fake, aligned device addresses; host-side checks
# reject the variations below before any CUDA call is made.
BASE = dict(q=0x10000, k=0x20000, v=0x20000, bt=0x30000, mbps=64, sl=0x40000, sel=0x50000, width=2048,
            seqs=8, rps=1, heads=64, bs=64, stride=64 * 512, ks=0.05, vs=0.05, sm=0.044, out=0x60000)


def _call(lib, **over):
    a = dict(BASE, **over)
    return lib.dsa_mla_decode(a["q"], a["k"], a["v"], a["bt"], a["mbps"], a["sl"], a["sel"], a["width"],
                              a["seqs"], a["rps"], a["heads"], a["bs"], a["stride"], a["ks"], a["vs"], a["sm"],
                              a["out"], None)


@pytest.mark.parametrize("over,code", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(bt=0), 1), (dict(sl=0), 1), (dict(sel=0), 1),
    (dict(out=0), 1), (dict(seqs=0), 1), (dict(heads=0), 1), (dict(rps=0), 1), (dict(bs=0), 1),
    (dict(width=0), 1), (dict(mbps=-1), 1), (dict(stride=64 * 512 - 16), 1), (dict(stride=64 * 512 + 8), 1),
    (dict(q=0x10008), 1), (dict(out=0x60002), 1), (dict(k=0x20004), 1), (dict(bt=0x30002), 1),
    (dict(width=8193), 2),
])
def test_invalid_arguments_rejected_on_host(lib, over, code):
    assert _call(lib, **over) == code


def _ws_args():
    a = BASE
    return [a["q"], a["k"], a["v"], a["bt"], a["mbps"], a["sl"], a["sel"], a["width"], a["seqs"], a["rps"],
            a["heads"], a["bs"], a["stride"], a["ks"], a["vs"], a["sm"], a["out"]]


def test_decode_ws_rejects_bad_workspace_on_host(lib):
    args = _ws_args()
    assert lib.dsa_mla_decode_ws(*args, 0, None, 1 << 20, None, None) == 1       # null workspace
    assert lib.dsa_mla_decode_ws(*args, 0, 0x70010, 1 << 20, None, None) == 1    # misaligned
    assert lib.dsa_mla_decode_ws(*args, 2, 0x70000, 1 << 20, None, None) == 1    # bad verify flag


@pytest.mark.parametrize("field,value", [("num_ctas", -1), ("tile_tokens", -1), ("tile_tokens", 1),
                                         ("tile_tokens", 32), ("tile_tokens", 96), ("tile_tokens", 256),
                                         ("gather_mode", -1), ("gather_mode", 3), ("reserved", 1)])
def test_decode_ws_rejects_bad_options_on_host(lib, field, value):
    o = _lib.DecodeOptions()
    setattr(o, field, value)
    assert lib.dsa_mla_decode_ws(*_ws_args(), 0, 0x70000, 1 << 20, ctypes.byref(o), None) == 1


def test_options_struct_matches_the_header():
    """The binding's struct has the header's fields, in order, with C layout."""
    text = open(_lib.HEADER).read()
    body = re.search(r"typedef struct dsa_decode_options \{(.*?)\} dsa_decode_options;", text, re.S).group(1)
    fields = re.findall(r"(\w+)\s*;", body)
    assert fields == [f for f, _ in _lib.DecodeOptions._fields_]
    assert ctypes.sizeof(_lib.DecodeOptions) == 40
    assert _lib.DecodeOptions.wait_limit_ns.offset == 16 and _lib.DecodeOptions.ev_begin.offset == 24


def test_resolve_rejects_bad_arguments_on_host(lib):
    assert lib.dsa_resolve_indices(None, 0x1000, 8, 1, 0x2000, 0x3000, None) == 1
    assert lib.dsa_resolve_indices(0x1000, 0x1000, 0, 1, 0x2000, 0x3000, None) == 1
    assert lib.dsa_resolve_indices(0x1000, 0x1000, 8, 0, 0x2000, 0x3000, None) == 1
    assert lib.dsa_resolve_indices(0x1002, 0x1000, 8, 1, 0x2000, 0x3000, None) == 1
    assert lib.dsa_resolve_indices(0x1000, 0x1000, 9000, 1, 0x2000, 0x3000, None) == 2


def test_workspace_size_grows_with_the_problem(lib):
    f = lib.dsa_mla_decode_workspace_bytes
    base = f(8, 1, 64, 2048, 152)
    assert base > 0 and base % 256 == 0
    assert f(16, 1, 64, 2048, 152) > base          # more rows
    assert f(8, 1, 128, 2048, 152) > base          # second head group
    assert f(8, 1, 64, 2048, 300) > base           # more partial slots
    # at least ids + byte offsets + counts + query images + f16 partials
    rows, width, ctas = 8, 2048, 152
    assert base >= rows * width * (4 + 8) + rows * 4 + rows * 65536 + 2 * ctas * 64 * 512 * 2
    assert f(0, 1, 64, 2048, 152) == 0



def test_explicit_grid_is_taken_as_given(lib):
    f = lib.dsa_mla_decode_grid
    assert f(128, 1, 128, 2048, 152) == 152
    assert f(1, 1, 4, 64, 7) == 7
    assert f(0, 1, 64, 2048, 152) == 0 and f(8, 1, 64, 2048, -1) == 0 and f(8, 1, 0, 2048, 1) == 0


def test_latent_write_rejects_bad_arguments_on_host(lib):
    f = lib.dsa_latent_write
    ok = dict(x=0x10000, w=0x20000, s=0x30000, rows=4, eps=1e-6, ks=0.05, bs=64, stride=64 * 512, c=0x40000)

    def call(**over):
        a = dict(ok, **over)
        return f(a["x"], a["w"], a["s"], a["rows"], a["eps"], a["ks"], a["bs"], a["stride"], a["c"], None)

    for over in (dict(x=0), dict(w=0), dict(s=0), dict(c=0), dict(rows=-1), dict(bs=0), dict(ks=0.0),
                 dict(eps=-1.0), dict(stride=64 * 512 - 16), dict(stride=64 * 512 + 8), dict(x=0x10004), dict(x=0x10008), dict(w=0x20008),
                 dict(s=0x30004), dict(c=0x40008)):
        assert call(**over) == 1, over
    assert call(rows=0) == 0                        # nothing to write: no device needed
    assert call(rows=0, x=0, s=0) == 0              # no rows: the row arrays may be null


def test_select_rejects_bad_arguments_on_host(lib):
    f = lib.dsa_select_pools
    ok = dict(sc=0x10000, q=0x20000, rows=4, n=100, kpool=4, topk=8, ids=0x30000)

    def call(**over):
        a = dict(ok, **over)
        return f(a["sc"], a["q"], a["rows"], a["n"], a["kpool"], a["topk"], a["ids"], None)

    for over in (dict(sc=0), dict(q=0), dict(ids=0), dict(rows=-1), dict(n=-1), dict(kpool=0), dict(topk=0),
                 dict(sc=0x10002), dict(q=0x20001), dict(ids=0x30002)):
        assert call(**over) == 1, over
    assert call(n=1 << 30, kpool=4) == 2            # token ids would pass 2^31
    assert call(topk=1 << 29, kpool=8) == 2
    assert call(rows=0, sc=0, q=0, ids=0) == 0       # nothing to select: no device needed


def test_absorb_rejects_bad_arguments_on_host(lib):
    for f in (lib.dsa_absorb_q, lib.dsa_absorb_o):
        ok = dict(a=0x10000, kv=0x20000, heads=4, nope=64, vd=64, kvl=512, other=256, out=0x30000, dt=0)

        def call(**over):
            a = dict(ok, **over)
            return f(a["a"], a["kv"], a["heads"], a["nope"], a["vd"], a["kvl"], a["other"], a["out"], a["dt"], None)

        for over in (dict(a=0), dict(kv=0), dict(out=0), dict(heads=0), dict(nope=0), dict(vd=0), dict(kvl=0),
                     dict(other=0), dict(dt=2), dict(dt=-1), dict(a=0x10001), dict(kv=0x20001), dict(out=0x30002)):
            assert call(**over) == 1, over
        assert call(heads=1 << 20, nope=1 << 11, vd=1 << 11) == 2     # heads*(nope+vd) past int

"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
function include/lla.h declares, and rejects invalid arguments before any launch."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

from looped_transformer_cross_gb300 import build, lla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return lla.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(lla_[a-z0-9_]+)\s*\(", txt))
    return sorted(names)


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert {"lla_encode", "lla_decode_attn", "lla_workspace_size", "lla_rope_table",
            "lla_device_status", "lla_status_string", "lla_abi_version"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    assert L.lla_abi_version() == 1


def test_status_strings(L):
    for s in range(7):
        assert lla.status_string(s) and lla.status_string(s) != "unknown status"
    assert lla.status_string(99) == "unknown status"


def test_workspace_size_rules(L):
    d = lla.dims(4, 16, 96, 160)
    n = lla.workspace_size(d, 32, 4096)
    assert n > 256
    # grows with batch; bf16 mode holds one query-operand image per (sequence, head)
    # (128 x r_k bf16 plus the 4 KB bias operand), fp32 mode the score buffer
    assert lla.workspace_size(d, 64, 4096) > n
    assert n >= 32 * 16 * (128 * 96 * 2 + 4096)
    n32 = lla.workspace_size(lla.dims(4, 16, 96, 160, dtype=lla.LLA_F32), 32, 4096)
    assert n32 >= 32 * 16 * 4096 * 4
    assert n32 - 32 * 16 * 4096 * 4 < n - 32 * 16 * (128 * 96 * 2 + 4096) + 256
    bad = lla.dims(4, 16, 96, 160, d_head=64)
    assert L.lla_workspace_size(ctypes.byref(bad), 1, 16, 0) == 0
    bad = lla.dims(4, 16, 90, 160)
    assert L.lla_workspace_size(ctypes.byref(bad), 1, 16, 0) == 0


def test_rope_table_is_fp64_rounded_once(L):
    d = lla.dims(4, 2, 16, 32, rope_base=10000.0)
    c, s = lla.rope_table(d, 5000)
    p = np.arange(5000)[:, None].astype(np.float64)
    theta = 10000.0 ** (-2.0 * np.arange(64) / 128.0)
    np.testing.assert_array_equal(c.numpy(), np.cos(p * theta).astype(np.float32))
    np.testing.assert_array_equal(s.numpy(), np.sin(p * theta).astype(np.float32))


def _null_call(L, dm, **over):
    args = dict(loop_t=0, q=None, B=1, L_max=128, rope_len=128, ws_bytes=1 << 20)
    args.update(over)
    cache = lla.Cache(None, None, args["B"], args["L_max"])
    return L.lla_decode_attn(ctypes.byref(dm), args["loop_t"], args["q"], cache, None, None, None,
                             None, None, None, None, None, args["rope_len"], None, None, None,
                             args["ws_bytes"], None)


def test_decode_rejects_bad_arguments_on_host(L):
    good = lla.dims(4, 2, 96, 160)
    assert _null_call(L, lla.dims(4, 2, 96, 160, d_head=64)) == lla.LLA_ERR_UNSUPPORTED
    assert _null_call(L, lla.dims(4, 2, 100, 160)) == lla.LLA_ERR_UNSUPPORTED
    assert _null_call(L, lla.dims(4, 2, 96, 272)) == lla.LLA_ERR_UNSUPPORTED
    assert _null_call(L, lla.dims(0, 2, 96, 160)) == lla.LLA_ERR_INVALID_ARG
    assert _null_call(L, lla.dims(4, 2, 96, 160, rope_base=-1.0)) == lla.LLA_ERR_INVALID_ARG
    assert _null_call(L, good, loop_t=4) == lla.LLA_ERR_INVALID_ARG
    assert _null_call(L, good, loop_t=-1) == lla.LLA_ERR_INVALID_ARG
    assert _null_call(L, good) == lla.LLA_ERR_INVALID_ARG          # null pointers
    assert _null_call(L, good, B=0) == lla.LLA_OK                   # nothing to do
    assert L.lla_decode_attn(None, 0, None, lla.Cache(None, None, 1, 1), None, None, None, None,
                             None, None, None, None, 1, None, None, None, 0, None) == lla.LLA_ERR_INVALID_ARG


def test_encode_rejects_bad_arguments_on_host(L):
    dm = lla.dims(4, 2, 96, 160)
    cache = lla.Cache(None, None, 1, 16)
    assert L.lla_encode(ctypes.byref(dm), None, None, 4, None, None, None, None, None, None, cache,
                        None, 0, None) == lla.LLA_ERR_INVALID_ARG
    assert L.lla_encode(ctypes.byref(dm), None, None, 0, None, None, None, None, None, None, cache,
                        None, 0, None) == lla.LLA_OK
    assert L.lla_encode(ctypes.byref(dm), None, None, -1, None, None, None, None, None, None, cache,
                        None, 0, None) == lla.LLA_ERR_INVALID_ARG


def test_misaligned_pointer_rejected(L):
    dm = lla.dims(1, 1, 16, 16)
    buf = (ctypes.c_char * 4096)()
    base = ctypes.addressof(buf)
    p = ctypes.c_void_p(base + (16 - base % 16) % 16 + 4)   # 4 bytes past a 16-byte boundary
    cache = lla.Cache(p, p, 1, 128)
    st = L.lla_decode_attn(ctypes.byref(dm), 0, p, cache, p, p, p, p, p, p, p, p, 128, p, p, p, 1 << 30, None)
    assert st == lla.LLA_ERR_INVALID_ARG


def test_decode_kernel_dispatch(L):
    """Which decode kernel family each shape takes (host-side decision, no launch)."""
    d = lambda *a, **k: lla.decode_kernel(lla.dims(*a, **k))
    assert d(4, 16, 16, 32) == "small-rank"          # Ouro-1.4B at rho = 21.3
    assert d(4, 2, 32, 64) == "small-rank"
    assert d(4, 6, 32, 64) == "small-rank"           # two epilogue groups (H mod 4 = 2)
    assert d(4, 8, 32, 32) == "small-rank"
    assert d(4, 8, 32, 64) == "tile"                 # four groups would get one slot each
    assert d(4, 16, 16, 64) == "tile"                # ring would be 2 slots
    assert d(4, 16, 32, 64) == "tile"                # 16 query images do not fit
    assert d(4, 3, 16, 32) == "tile"                 # odd H
    assert d(4, 18, 16, 32) == "tile"                # more heads than resident images
    assert d(4, 16, 96, 160) == "tile"
    assert d(4, 16, 48, 80) == "tile"
    assert d(4, 16, 128, 256, variant=lla.LLA_2D) == "pair-2d"
    assert d(4, 16, 16, 32, dtype=lla.LLA_F32) == "fp32"
    assert d(4, 16, 16, 32, d_head=64) is None


def test_decoupled_kernel_dispatch(L):
    """Which decoupled-RoPE kernel family each shape takes (host-side, no launch)."""
    d = lambda *a, d_rope=64, **k: lla.decoupled_kernel(lla.dims(*a, **k), d_rope)
    assert d(4, 16, 16, 32) == "small-rank"          # Ouro-1.4B at rho = 21.3
    assert d(4, 16, 32, 64) == "small-rank"
    assert d(4, 2, 16, 64) == "small-rank"
    assert d(4, 6, 32, 32) == "small-rank"           # three heads per epilogue group
    assert d(4, 3, 16, 32) == "tile"                 # odd H
    assert d(4, 18, 16, 32) == "tile"                # more heads than resident images
    assert d(4, 16, 48, 80) == "tile"
    assert d(4, 16, 96, 160) == "tile"               # Ouro-1.4B at rho = 4
    assert d(4, 16, 16, 32, dtype=lla.LLA_F32) == "fp32"
    assert d(4, 16, 16, 32, d_rope=32) is None
    assert d(4, 16, 16, 32, variant=lla.LLA_2D) is None
    assert d(4, 16, 256, 256) is None                # r_k above the tile kernel's 128
    assert d(4, 16, 128, 256) == "tile"              # the tile kernel's largest ranks
    assert d(4, 16, 144, 160) is None


def test_decoupled_workspace_sizes(L):
    """Workspace bytes of the decoupled call: the tensor-core kernels' records, images,
    sc b0 and cos/sin table grow with the batch and the context; bf16 shapes no kernel
    takes report 0 (the call returns LLA_ERR_UNSUPPORTED); fp32 mode holds the scores."""
    ws = lambda *a, B=32, L_max=4096, **k: L.lla_decoupled_workspace_size(ctypes.byref(lla.dims(*a, **k)), 64, B, L_max)
    small, tile = ws(4, 16, 16, 32), ws(4, 16, 96, 160)
    assert small > 0 and tile > 0
    # B images of 4 KB + 512 B per 16 K-latent columns, for every (sequence, head)
    assert tile - ws(4, 16, 96, 160, B=31) >= 16 * (4096 + 6 * 512)
    assert ws(4, 16, 96, 160, L_max=8192) > tile                      # cos/sin table rows
    assert ws(4, 16, 144, 160) == 0
    assert ws(4, 16, 96, 160, dtype=lla.LLA_F32) >= 256 + 32 * 16 * 4096 * 4   # scores
    assert L.lla_decoupled_workspace_size(ctypes.byref(lla.dims(4, 16, 96, 160)), 32, 32, 4096) == 0


def test_window_rejects_bad_arguments_on_host(L):
    dm = lla.dims(4, 2, 16, 32)
    call = lambda d, B=1, W=8, rope_len=128, ws=1 << 20: L.lla_window_attn(
        ctypes.byref(d), B, W, None, None, None, None, None, None, None, None, rope_len, None, None, None, ws, None)
    assert call(dm) == lla.LLA_ERR_INVALID_ARG                       # null pointers
    assert call(dm, B=-1) == lla.LLA_ERR_INVALID_ARG
    assert call(dm, W=-1) == lla.LLA_ERR_INVALID_ARG
    assert call(dm, rope_len=0) == lla.LLA_ERR_INVALID_ARG
    assert call(dm, rope_len=127) == lla.LLA_ERR_INVALID_ARG
    assert call(lla.dims(4, 2, 16, 32, d_head=64)) == lla.LLA_ERR_UNSUPPORTED
    assert call(dm, B=0) == lla.LLA_OK                               # nothing to do
    assert call(dm, W=0) == lla.LLA_OK


def test_paged_rejects_bad_arguments_on_host(L):
    """lla_decode_attn_paged / lla_encode_paged: host checks of the page description
    (no launch)."""
    tbl = (ctypes.c_int32 * 64)()
    good_bt = ctypes.c_void_p(ctypes.addressof(tbl))

    def dec(dm, page_size=128, max_pages=4, num_pages=8, B=1, bt=good_bt):
        cache = lla.PagedCache(None, None, bt, B, max_pages, page_size, num_pages)
        return L.lla_decode_attn_paged(ctypes.byref(dm), 0, None, cache, None, None, None, None, None, None,
                                       None, None, 1024, None, None, None, 1 << 20, None)

    def enc(dm, page_size=128):
        cache = lla.PagedCache(None, None, good_bt, 1, 4, page_size, 8)
        return L.lla_encode_paged(ctypes.byref(dm), None, None, 4, None, None, None, None, None, None, cache,
                                  None, 1 << 20, None)

    bf16, f32 = lla.dims(4, 2, 96, 160), lla.dims(4, 2, 96, 160, dtype=lla.LLA_F32)
    assert dec(lla.dims(4, 2, 96, 160, variant=lla.LLA_2D)) == lla.LLA_ERR_UNSUPPORTED
    assert dec(bf16, bt=None) == lla.LLA_ERR_INVALID_ARG
    assert dec(bf16, bt=ctypes.c_void_p(ctypes.addressof(tbl) + 2)) == lla.LLA_ERR_INVALID_ARG
    assert dec(bf16, max_pages=0) == lla.LLA_ERR_INVALID_ARG
    assert dec(bf16, num_pages=0) == lla.LLA_ERR_INVALID_ARG
    assert dec(bf16, page_size=0) == lla.LLA_ERR_INVALID_ARG
    assert dec(bf16, B=0) == lla.LLA_OK                              # nothing to do
    # any page size passes the page checks, in both storage types (then the call fails
    # on the null pointers)
    for P in (1, 8, 16, 64, 100, 128, 256):
        assert dec(bf16, page_size=P) == lla.LLA_ERR_INVALID_ARG
        assert dec(f32, page_size=P) == lla.LLA_ERR_INVALID_ARG
        assert enc(bf16, page_size=P) == lla.LLA_ERR_INVALID_ARG
    assert dec(bf16, page_size=1, B=0) == lla.LLA_OK
    assert dec(f32, page_size=1, B=0) == lla.LLA_OK


def test_evict_rejects_bad_arguments_on_host(L):
    buf = (ctypes.c_char * 1024)()
    base = ctypes.addressof(buf)
    p = ctypes.c_void_p(base + (16 - base % 16) % 16)
    dm = lla.dims(4, 2, 96, 160)

    def call(sink=4, window=256, B=1, ptr=p, ws=256, d=dm):
        cache = lla.Cache(ptr, ptr, B, 300)
        return L.lla_evict_window(ctypes.byref(d), cache, ptr, sink, window, ptr, ws, None)

    assert call(sink=-1) == lla.LLA_ERR_INVALID_ARG
    assert call(window=-1) == lla.LLA_ERR_INVALID_ARG
    assert call(sink=0, window=0) == lla.LLA_ERR_INVALID_ARG        # an empty budget
    assert call(B=-1) == lla.LLA_ERR_INVALID_ARG
    assert call(ptr=None) == lla.LLA_ERR_INVALID_ARG
    assert call(ptr=ctypes.c_void_p(p.value + 4)) == lla.LLA_ERR_INVALID_ARG
    assert call(ws=255) == lla.LLA_ERR_INVALID_ARG
    assert call(d=lla.dims(4, 2, 96, 160, d_head=64)) == lla.LLA_ERR_UNSUPPORTED
    assert call(B=0) == lla.LLA_OK                                  # nothing to do


def declared_arity():
    """Parameter count of every function include/lla.h declares (void lists count 0)."""
    out = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        txt = open(os.path.join(ROOT, "include", fn)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        for name, params in re.findall(r"\b(lla_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", txt, flags=re.S):
            p = params.strip()
            out[name] = 0 if p in ("", "void") else p.count(",") + 1
    return out


def test_binding_signatures_match_the_header(L):
    """Every function the header declares has a ctypes signature in the binding, with as
    many arguments as the header's prototype (a drift here would pass garbage through
    the ABI)."""
    arity = declared_arity()
    assert set(arity) == set(declared_functions())
    for name, n in arity.items():
        f = getattr(L, name)
        assert f.argtypes is not None, name + " has no ctypes signature in the binding"
        assert len(f.argtypes) == n, (name, len(f.argtypes), n)


def _declared_params():
    """(name, [parameter declaration]) of every prototype in include/lla.h."""
    out = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        txt = open(os.path.join(ROOT, "include", fn)).read()
        txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
        for name, params in re.findall(r"\b(lla_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", txt, flags=re.S):
            p = " ".join(params.split())
            out[name] = [] if p in ("", "void") else [x.strip() for x in p.split(",")]
    return out


def test_binding_argument_types_match_the_header(L):
    """Each argument's ctypes type agrees with the header's C type: pointers as pointers,
    int as a 32-bit int, int64_t and size_t as 64-bit, the cache descriptors by value."""
    by_value = {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
                "float": ctypes.c_float, "lla_status": ctypes.c_int, "lla_cache": lla.Cache,
                "lla_paged_cache": lla.PagedCache}
    ints = (ctypes.c_int, ctypes.c_uint, ctypes.c_long, ctypes.c_ulong, ctypes.c_longlong,
            ctypes.c_ulonglong)

    def same(ct, want):
        return ct is want or (ct in ints and want in ints and ctypes.sizeof(ct) == ctypes.sizeof(want))

    for name, params in _declared_params().items():
        f = getattr(L, name)
        for i, (decl, ct) in enumerate(zip(params, f.argtypes)):
            if "*" in decl:
                assert ct is ctypes.c_void_p or issubclass(ct, ctypes._Pointer), (name, i, decl, ct)
            else:
                want = by_value[decl.replace("const ", "").split()[0]]
                assert same(ct, want), (name, i, decl, ct)


def test_struct_layouts_match_the_header(tmp_path):
    """The binding's ctypes structures have the C structures' size and field offsets, as
    gcc lays them out from include/lla.h (they cross the ABI by value or by pointer)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    specs = {"lla_dims": (lla.Dims, ["T", "H", "d_head", "r_k", "r_v", "variant", "dtype", "rope_base",
                                     "rope_style"]),
             "lla_cache": (lla.Cache, ["k", "v", "B", "L_max"]),
             "lla_paged_cache": (lla.PagedCache, ["k", "v", "block_table", "B", "max_pages", "page_size",
                                                  "num_pages"])}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "lla.h"', "int main(void) {"]
    for cname, (_, fields) in specs.items():
        lines.append('printf("%s size %%zu\\n", sizeof(%s));' % (cname, cname))
        for f in fields:
            lines.append('printf("%s %s %%zu\\n", offsetof(%s, %s));' % (cname, f, cname, f))
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([str(exe)], capture_output=True, text=True,
                                                              check=True).stdout.splitlines())
    for cname, (cls, fields) in specs.items():
        assert int(got["%s size" % cname]) == ctypes.sizeof(cls), cname
        for f in fields:
            assert int(got["%s %s" % (cname, f)]) == getattr(cls, f).offset, (cname, f)


def test_enum_constants_match_the_header():
    """Every enumerator of include/lla.h that the binding names has the header's value, and
    the binding names every status code."""
    txt = open(os.path.join(ROOT, "include", "lla.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    values = {n: int(v) for n, v in re.findall(r"\b(LLA_[A-Z0-9_]+)\s*=\s*(\d+)", txt)}
    statuses = [n for n in values if n == "LLA_OK" or n.startswith("LLA_ERR_")]
    assert len(statuses) == 7
    for n in statuses:
        assert hasattr(lla, n), n
    for n, v in values.items():
        if hasattr(lla, n):
            assert getattr(lla, n) == v, n

"""The C-ABI library loads, exports every entry point its header declares, and rejects bad arguments on
the host (before any device work), all without a GPU."""
import ctypes
import os
import re

import pytest

import decode_attention_19_b300 as L
from decode_attention_19_b300 import binding as Bd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lowram.h")


def declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"LOWRAM_API\s+[\w\s\*]+?\b(lowram_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol():
    names = declared()
    assert len(names) >= 12, names
    lib = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in lowram.h but not exported"


def test_status_strings_and_version():
    lib = L.lib()
    for st in range(7):
        assert lib.lowram_status_string(st)
    assert L.lowram_version() >= 100


def shape(**kw):
    base = dict(B=8, T=8192, H_q=32, H_kv=8, d=128, r=512, m=128, S=1024, n_res=820, act_dtype=1, coef_dtype=1,
                res_dtype=1, max_pos=8192, sm_scale=0.0)
    base.update(kw)
    return L.lowram_decode_shape(*[base[f] for f, _ in L.lowram_decode_shape._fields_])


def test_workspace_size_covers_scratch():
    n = L.lowram_decode_workspace_size(shape())
    B, Hkv, T, S, Hq, d = 8, 8, 8192, 1024, 32, 128
    assert n % 256 == 0
    assert n >= 4 * B * Hkv * T + 4 * B * Hkv * S + 4 * B * Hq * (d + 2)


@pytest.mark.parametrize("kw,status", [
    (dict(H_q=30), 1), (dict(d=96), 3), (dict(r=500), 3), (dict(m=300), 3), (dict(n_res=9000), 1),
    (dict(act_dtype=7), 1), (dict(coef_dtype=0), 3), (dict(res_dtype=9), 1), (dict(B=-1), 1),
    (dict(H_q=72, H_kv=8), 3), (dict(max_pos=0), 1),
])
def test_bad_shapes_are_rejected(kw, status):
    with pytest.raises(Bd.LowramError) as ei:
        L.lowram_decode_workspace_size(shape(**kw))
    assert ei.value.status == status


def _call(s, ptrs, ws_bytes=1 << 30):
    lib = L.lib()
    args = [ctypes.c_void_p(p) if p else None for p in ptrs]
    return lib.lowram_decode_attn(ctypes.byref(s), *args, ctypes.c_void_p(0x10000000), ws_bytes, None)


def test_decode_rejects_misaligned_and_missing_pointers_on_host():
    s = shape()
    good = [0x1000 * (i + 1) for i in range(18)]
    # order: q coef coef_scale pos cos sin basis w1 w2 b1 b2 res_idx res_val res_scale out lse sel key
    ptrs = list(good)
    ptrs[1] = 0x2008                       # misaligned coef
    assert _call(s, ptrs) == 2
    ptrs = list(good)
    ptrs[0] = 0                            # q missing
    assert _call(s, ptrs) == 1
    ptrs = list(good)
    ptrs[11] = 0                           # residual list missing while n_res > 0
    assert _call(s, ptrs) == 1
    assert _call(s, good, ws_bytes=1024) == 4   # workspace too small
    assert "workspace" in L.lib().lowram_last_error().decode()


def test_compress_and_dense_shape_checks():
    cs = L.lowram_compress_shape(8, 8192, 4, 8, 128, 512, 128, 820, 1, 1, 1, 0, 0)
    assert L.lowram_compress_workspace_size(cs) >= 4 * 8 * 8 * 8192
    bad = L.lowram_compress_shape(8, 8192, 17, 8, 128, 512, 128, 820, 1, 1, 1, 0, 0)
    with pytest.raises(Bd.LowramError):
        L.lowram_compress_workspace_size(bad)
    assert L.lowram_dense_workspace_size(8, 8192, 32, 8, 128) > 0
    with pytest.raises(Bd.LowramError):
        L.lowram_dense_workspace_size(8, 8192, 30, 8, 128)


def test_rope_table_rejects_bad_arguments():
    lib = L.lib()
    assert lib.lowram_rope_table(7, 1e4, 10, None, None, None) == 1
    assert lib.lowram_rope_table(8, -1.0, 10, None, None, None) == 1
    assert lib.lowram_rope_table(8, 1e4, 0, None, None, None) == 0

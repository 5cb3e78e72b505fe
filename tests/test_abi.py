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
                res_dtype=1, max_pos=8192, sm_scale=0.0, basis_batch_stride=0, mlp_batch_stride=0, flags=0)
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


def test_tail_merge_and_fit_entry_points_check_arguments_on_the_host():
    """Host-side argument checks of the exact tail, the merge, the fitted basis and the predictor fit: each
    rejects a bad argument with its status before any device work (no GPU needed)."""
    import ctypes
    lib = L.lib()
    INVALID, UNSUPPORTED, WORKSPACE = 1, 3, 4
    # tail append: row outside the capacity, bad head dim, bad dtype
    assert lib.lowram_tail_append(2, 8, 2, 128, 1, 8, None, None, None, None, None) == INVALID
    assert lib.lowram_tail_append(2, 8, 2, 96, 1, 0, None, None, None, None, None) == INVALID
    assert lib.lowram_tail_append(2, 8, 2, 128, 7, 0, None, None, None, None, None) == INVALID
    assert lib.lowram_tail_append(0, 8, 2, 128, 1, 0, None, None, None, None, None) == 0     # nothing to do
    # tail attention: length past the capacity
    assert lib.lowram_tail_decode_attn(2, 8, 9, 8, 2, 128, 1, 0.0, None, None, None, None, None, None, 0,
                                       None) == INVALID
    # merge: missing operands
    assert lib.lowram_merge_attn(2, 8, 128, None, None, None, None, None, None, None) == INVALID
    assert lib.lowram_merge_attn(0, 8, 128, None, None, None, None, None, None, None) == 0
    # fitted basis: rank above G*H_kv*d, fewer tokens than the rank, rank not a multiple of 32
    n = ctypes.c_size_t(0)
    assert lib.lowram_fit_basis_workspace_size(ctypes.byref(L.lowram_compress_shape(2, 100, 1, 1, 64, 96, 32, 0, 1, 1,
                                                                                    1, 0, 0)), ctypes.byref(n)) == UNSUPPORTED
    assert lib.lowram_fit_basis_workspace_size(ctypes.byref(L.lowram_compress_shape(1, 20, 2, 2, 64, 32, 32, 0, 1, 1,
                                                                                    1, 0, 0)), ctypes.byref(n)) == INVALID
    assert lib.lowram_fit_basis_workspace_size(ctypes.byref(L.lowram_compress_shape(2, 100, 2, 2, 64, 40, 32, 0, 1, 1,
                                                                                    1, 0, 0)), ctypes.byref(n)) == UNSUPPORTED
    good = L.lowram_compress_shape(8, 8192, 4, 8, 128, 512, 128, 0, 1, 1, 1, 0, 0)
    assert lib.lowram_fit_basis_workspace_size(ctypes.byref(good), ctypes.byref(n)) == 0
    assert n.value >= 4 * 8 * 8192 * 4096 + 4 * 4096 * 4096       # the float32 keys and the Gram matrix
    assert lib.lowram_fit_basis(ctypes.byref(good), None, None, None, None, 8, 0, None, None, None, 0,
                                None) == WORKSPACE
    # predictor fit: hidden width, head dim, Adam hyper-parameters, workspace
    assert lib.lowram_fit_predictor_workspace_size(1, 10, 8, 128, 300, ctypes.byref(n)) == UNSUPPORTED
    assert lib.lowram_fit_predictor_workspace_size(1, 10, 8, 96, 128, ctypes.byref(n)) == UNSUPPORTED
    assert lib.lowram_fit_predictor_workspace_size(1, 10, 8, 128, 128, ctypes.byref(n)) == 0
    assert n.value >= 3 * 4 * 8 * (2 * 128 * 128 + 256)      # gradient and the two moments
    n_big = ctypes.c_size_t(0)
    assert lib.lowram_fit_predictor_workspace_size(8, 8192, 8, 128, 128, ctypes.byref(n_big)) == 0
    assert n_big.value >= 12 * 8 * 8192 * 8 * 128              # the keys' bf16 terms in two layouts
    ws = ctypes.create_string_buffer(n.value + 256)
    wsp = ctypes.c_void_p((ctypes.addressof(ws) + 255) & ~255)
    assert lib.lowram_fit_predictor(1, 10, 8, 128, 128, 1, None, None, 5, 0.0, 0.9, 0.999, 1e-8, None, None, None,
                                    None, None, wsp, n.value, None) == INVALID                    # lr <= 0
    assert lib.lowram_fit_predictor(1, 10, 8, 128, 128, 1, None, None, 5, 1e-3, 1.0, 0.999, 1e-8, None, None, None,
                                    None, None, wsp, n.value, None) == INVALID                    # beta1 = 1
    assert lib.lowram_fit_predictor(1, 10, 8, 128, 128, 1, None, None, 5, 1e-3, 0.9, 0.999, 1e-8, None, None, None,
                                    None, None, None, 0, None) == WORKSPACE
    assert lib.lowram_predictor_grad(1, 10, 8, 128, 128, 1, None, None, None, None, None, None, None, None, None, None,
                                     None, None) == INVALID


def test_eviction_entry_points_and_batch_limit_check_arguments_on_the_host():
    """Host-side checks of the attention mass and the eviction plan (shape, dtype, window, workspace, the plan's
    budget) and of the per-call batch limit shared by the kernels with one grid row per sequence."""
    import ctypes
    lib = L.lib()
    INVALID, UNSUPPORTED, WORKSPACE = 1, 3, 4
    n = ctypes.c_size_t(0)
    # attention mass: empty window, head ratio 3, head dim 96, bad dtype, batch above the grid limit
    assert lib.lowram_attention_mass_workspace_size(2, 100, 0, 32, 8, 128, 1, ctypes.byref(n)) == INVALID
    assert lib.lowram_attention_mass_workspace_size(2, 100, 4, 24, 8, 128, 1, ctypes.byref(n)) == UNSUPPORTED
    assert lib.lowram_attention_mass_workspace_size(2, 100, 4, 32, 8, 96, 1, ctypes.byref(n)) == UNSUPPORTED
    assert lib.lowram_attention_mass_workspace_size(2, 100, 4, 32, 8, 128, 7, ctypes.byref(n)) == INVALID
    assert lib.lowram_attention_mass_workspace_size(65536, 100, 4, 32, 8, 128, 1, ctypes.byref(n)) == UNSUPPORTED
    # bf16 scratch: the log-sum-exps, the chunks' (max, sum) pairs and the packed window queries
    assert lib.lowram_attention_mass_workspace_size(4, 65536, 32, 32, 8, 128, 1, ctypes.byref(n)) == 0
    assert n.value >= 4 * 4 * 32 * 32 + 2 * 4 * 8 * 128 * 128
    bf16_bytes = n.value
    assert lib.lowram_attention_mass_workspace_size(4, 65536, 32, 32, 8, 128, 0, ctypes.byref(n)) == 0
    assert n.value >= 4 * 4 * 32 * 32 and n.value != bf16_bytes
    assert lib.lowram_attention_mass(4, 100, 32, 32, 8, 128, 1, 0.0, None, None, None, None, 0, None) == WORKSPACE
    ws = ctypes.create_string_buffer((1 << 21) + 256)
    wsp = ctypes.c_void_p((ctypes.addressof(ws) + 255) & ~255)
    assert lib.lowram_attention_mass(0, 100, 32, 32, 8, 128, 1, 0.0, None, None, None, wsp, 1 << 21, None) == 0
    assert lib.lowram_attention_mass(2, 100, 4, 32, 8, 128, 1, 0.0, None, None, None, wsp, 1 << 21, None) == INVALID
    # eviction plan: budget above T, forced tokens above the budget, workspace
    assert lib.lowram_evict_plan_workspace_size(2, 100, ctypes.byref(n)) == 0
    assert n.value >= 4 * 2 * 100
    assert lib.lowram_evict_plan(2, 100, 4, 8, 101, None, None, wsp, n.value, None) == INVALID
    assert lib.lowram_evict_plan(2, 100, 40, 40, 60, None, None, wsp, n.value, None) == INVALID
    assert lib.lowram_evict_plan(2, 100, 4, 8, 50, None, None, None, 0, None) == WORKSPACE
    # the batch limit on the other entry points with one grid row per sequence
    assert lib.lowram_dense_workspace_size(65536, 100, 32, 8, 128, ctypes.byref(n)) == UNSUPPORTED
    assert lib.lowram_dense_workspace_size(65535, 100, 32, 8, 128, ctypes.byref(n)) == 0
    # and on the token rows: B*T below 2^31
    assert lib.lowram_attention_mass_workspace_size(2, 1 << 30, 1, 8, 8, 64, 1, ctypes.byref(n)) == UNSUPPORTED
    assert lib.lowram_fit_predictor_workspace_size(2, 1 << 30, 8, 128, 128, ctypes.byref(n)) == UNSUPPORTED
    # the predictor fit's own limit: 65535 * 32 prompt tokens (the split passes' grid rows)
    assert lib.lowram_fit_predictor_workspace_size(1, 65535 * 32, 8, 128, 128, ctypes.byref(n)) == 0
    assert lib.lowram_fit_predictor_workspace_size(1, 65535 * 32 + 1, 8, 128, 128, ctypes.byref(n)) == UNSUPPORTED
    assert lib.lowram_predictor_grad(2, 1 << 30, 8, 128, 128, 1, None, None, None, None, None, None, None, None, None,
                                     None, None, None) == UNSUPPORTED


def test_wait_limit_is_checked_on_the_host():
    with pytest.raises(Bd.LowramError) as ei:
        L.lowram_set_wait_limit(-1)
    assert ei.value.status == 1
    L.lowram_set_wait_limit(0)          # the default


def test_batch_strides_are_checked_and_size_the_workspace():
    per = 8 * 128 * 512
    for kw in (dict(basis_batch_stride=per - 8), dict(basis_batch_stride=per + 4), dict(basis_batch_stride=-8),
               dict(mlp_batch_stride=8 * 128 * 128 - 8), dict(mlp_batch_stride=8 * 128 * 128 + 2)):
        with pytest.raises(Bd.LowramError) as ei:
            L.lowram_decode_workspace_size(shape(**kw))
        assert ei.value.status == 1, kw
    shared = L.lowram_decode_workspace_size(shape())
    own = L.lowram_decode_workspace_size(shape(basis_batch_stride=per, mlp_batch_stride=8 * 128 * 128))
    if L.lowram_decode_uses_tensor_cores(shape()):    # (needs the driver's tensor-map encoder)
        # one folded first layer [H_kv, m, r] bf16 per sequence instead of one for all
        assert own - shared >= 7 * 8 * 128 * 512 * 2
    else:
        assert own == shared


def test_check_word_bits_match_the_header():
    import re
    import decode_attention_19_b300 as L
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lowram.h")).read()
    bits = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define LOWRAM_CHECK_(\w+) (\d+)u", hdr)}
    assert bits == {"POS_RANGE": 1, "RES_INDEX": 2, "TIMEOUT": 4, "NOT_PD": 8, "LAYOUT": 16}
    for name, v in bits.items():
        assert getattr(L, "CHECK_" + name) == v

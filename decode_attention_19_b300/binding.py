"""Thin ctypes binding of liblowram.so.  Argument marshalling only: every step of the path runs in the
library's CUDA kernels; this module reads shapes and dtypes off torch tensors, allocates outputs and
workspaces with torch, and passes raw device pointers and the current CUDA stream.

The functions carry the names of the C entry points in include/lowram.h.  If the library is not
built the first call raises (there is no other implementation to fall back to).

Example: one layer group of a prefilled prompt, then a decode step (all tensors on the GPU; shapes as in
include/lowram.h)::

    import torch
    import decode_attention_19_b300 as L

    B, T, G, H_q, H_kv, d, r, m = 2, 2048, 4, 32, 8, 128, 512, 128
    dev, bf = "cuda", torch.bfloat16
    keys = torch.randn(B, T, G, H_kv, d, device=dev).to(bf)            # the G layers' pre-RoPE keys
    values = [torch.randn(B, T, H_kv, d, device=dev).to(bf) for _ in range(G)]

    # fit the group's shared key basis, and each layer's value predictor (float32 master copies)
    proj, bases, _ = L.lowram_fit_basis(keys, r)
    W1, B1, W2, B2 = [], [], [], []
    for l in range(G):
        w1, b1 = torch.randn(H_kv, m, d, device=dev) * d ** -0.5, torch.zeros(H_kv, m, device=dev)
        w2, b2 = torch.randn(H_kv, d, m, device=dev) * m ** -0.5, torch.zeros(H_kv, d, device=dev)
        L.lowram_fit_predictor(keys[:, :, l].contiguous(), values[l], w1, b1, w2, b2, steps=50, lr=1e-3)
        W1.append(w1.to(bf))
        W2.append(w2.to(bf))
        B1.append(b1)
        B2.append(b2)

    # write the compressed cache: latent coefficients shared by the group, residuals for the worst 10 % per layer
    cache = L.lowram_compress(keys, values, proj, bases, W1, W2, n_res=T // 10, coef_dtype=L.LOWRAM_BF16,
                              res_dtype=L.LOWRAM_BF16, b1s=B1, b2s=B2)

    # one decode step of layer l: attend the compressed body, then the exact tail of tokens decoded since
    l = 0
    cos, sin = L.lowram_rope_table(d, 5e5, T + 256)
    q = torch.randn(B, H_q, d, device=dev).to(bf)                      # already rotated at its position
    out, lse = L.lowram_decode_attn(q, cache["coef"], bases[l], W1[l], W2[l], rope_cos=cos, rope_sin=sin, S=512,
                                    b1=B1[l], b2=B2[l], res_idx=cache["res_idx"][l], res_val=cache["res_val"][l])
    tail_k = torch.zeros(B, 256, H_kv, d, device=dev, dtype=bf)
    tail_v = torch.zeros_like(tail_k)
    L.lowram_tail_append(torch.randn(B, H_kv, d, device=dev).to(bf), torch.randn(B, H_kv, d, device=dev).to(bf),
                         tail_k, tail_v, 0)
    out_t, lse_t = L.lowram_tail_decode_attn(q, tail_k, tail_v, 1)
    out, lse = L.lowram_merge_attn(out, lse, out_t, lse_t)
    assert L.lowram_get_error(cache["workspace"]) == 0               # no out-of-range data seen by the kernels

    # an evicted cache: choose the kept tokens from the last 32 queries' attention, then compress only those
    q_window = torch.randn(B, 32, H_q, d, device=dev).to(bf)
    k_rotated = torch.randn(B, T, H_kv, d, device=dev).to(bf)
    keep = L.lowram_evict_plan(L.lowram_attention_mass(q_window, k_rotated), n_sink=64, n_recent=256, T_keep=T // 4)
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblowram.so")

LOWRAM_F32, LOWRAM_BF16, LOWRAM_INT4_G32, LOWRAM_INT8_VEC = 0, 1, 2, 3
CHECK_POS_RANGE, CHECK_RES_INDEX, CHECK_TIMEOUT, CHECK_NOT_PD, CHECK_LAYOUT = 1, 2, 4, 8, 16
FLAG_INT4_EXACT_SPLIT = 1
STATUS = {0: "ok", 1: "invalid argument", 2: "alignment", 3: "unsupported", 4: "workspace", 5: "cuda",
          6: "device check"}


class lowram_decode_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "T", "H_q", "H_kv", "d", "r", "m", "S", "n_res", "act_dtype",
                                              "coef_dtype", "res_dtype", "max_pos")] + [("sm_scale", ctypes.c_float)] + \
        [("basis_batch_stride", ctypes.c_int64), ("mlp_batch_stride", ctypes.c_int64), ("flags", ctypes.c_uint32)]


class lowram_compress_shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "T", "G", "H_kv", "d", "r", "m", "n_res", "act_dtype", "coef_dtype",
                                              "res_dtype", "keys_post_rope", "max_pos")]


class LowramError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"liblowram: {STATUS.get(status, status)}: {msg}")
        self.status = status


class LowramShapeError(ValueError):
    """A tensor is smaller than the layout its call reads or writes, or holds elements of another size.  The C
    entry points see pointers and sizes only, so the binding checks every buffer against the sizes it passes."""


_ESZ = {LOWRAM_F32: 4, LOWRAM_BF16: 2}


def _need(name: str, t: Optional[torch.Tensor], numel: int, itemsize: int):
    """t (if given) holds at least `numel` elements of `itemsize` bytes."""
    if t is None:
        return
    if t.element_size() != itemsize:
        raise LowramShapeError(f"{name}: elements of {itemsize} bytes expected, got {t.dtype}")
    if t.numel() < numel:
        raise LowramShapeError(f"{name}: at least {numel} elements expected, got shape {tuple(t.shape)}")


def _need_list(name: str, ts, n: int, numel: int, itemsize: int):
    if ts is None:
        return
    if len(ts) != n:
        raise LowramShapeError(f"{name}: {n} tensors expected, got {len(ts)}")
    for i, t in enumerate(ts):
        _need(f"{name}[{i}]", t, numel, itemsize)


_lib = None
_vp = ctypes.c_void_p


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -m decode_attention_19_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        i32, sz, dbl, flt = ctypes.c_int32, ctypes.c_size_t, ctypes.c_double, ctypes.c_float
        psz = ctypes.POINTER(ctypes.c_size_t)
        sigs = {
            "lowram_decode_workspace_size": [ctypes.POINTER(lowram_decode_shape), psz],
            "lowram_decode_attn": [ctypes.POINTER(lowram_decode_shape)] + [_vp] * 18 + [_vp, sz, _vp],
            "lowram_decode_attn_events": [ctypes.POINTER(lowram_decode_shape)] + [_vp] * 18 + [_vp, sz, _vp, _vp],
            "lowram_decode_attn_static": [ctypes.POINTER(lowram_decode_shape)] + [_vp] * 18 + [_vp],
            "lowram_decode_attn_static_get_error": [_vp, ctypes.POINTER(ctypes.c_uint32)],
            "lowram_rope_table": [i32, dbl, i32, _vp, _vp, _vp],
            "lowram_compress_workspace_size": [ctypes.POINTER(lowram_compress_shape), psz],
            "lowram_compress": [ctypes.POINTER(lowram_compress_shape)] + [_vp] * 18 + [sz, _vp],
            "lowram_dense_workspace_size": [i32, i32, i32, i32, i32, psz],
            "lowram_dense_decode_attn": [i32, i32, i32, i32, i32, i32, flt, _vp, _vp, _vp, _vp, _vp, _vp, sz, _vp],
            "lowram_attention_mass_workspace_size": [i32] * 7 + [psz],
            "lowram_attention_mass": [i32] * 7 + [flt, _vp, _vp, _vp, _vp, sz, _vp],
            "lowram_evict_plan_workspace_size": [i32, i32, psz],
            "lowram_evict_plan": [i32] * 5 + [_vp, _vp, _vp, sz, _vp],
            "lowram_predictor_grad": [i32] * 6 + [_vp] * 11 + [_vp],
            "lowram_fit_predictor_workspace_size": [i32] * 5 + [psz],
            "lowram_fit_predictor": [i32] * 6 + [_vp, _vp, i32, flt, flt, flt, flt] + [_vp] * 6 + [sz, _vp],
            "lowram_fit_basis_workspace_size": [ctypes.POINTER(lowram_compress_shape), psz],
            "lowram_fit_basis": [ctypes.POINTER(lowram_compress_shape), _vp, _vp, _vp, _vp, i32, ctypes.c_uint64, _vp,
                                 _vp, _vp, sz, _vp],
            "lowram_tail_append": [i32, i32, i32, i32, i32, i32, _vp, _vp, _vp, _vp, _vp],
            "lowram_tail_decode_attn": [i32, i32, i32, i32, i32, i32, i32, flt, _vp, _vp, _vp, _vp, _vp, _vp, sz, _vp],
            "lowram_merge_attn": [i32, i32, i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
            "lowram_get_error": [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)],
            "lowram_decode_uses_tensor_cores": [ctypes.POINTER(lowram_decode_shape), ctypes.POINTER(ctypes.c_int32)],
            "lowram_clear_error": [_vp, _vp],
            "lowram_set_wait_limit": [ctypes.c_int64],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.lowram_status_string.restype = ctypes.c_char_p
        L.lowram_status_string.argtypes = [ctypes.c_int]
        L.lowram_last_error.restype = ctypes.c_char_p
        L.lowram_last_error.argtypes = []
        L.lowram_version.restype = ctypes.c_int32
        _lib = L
    return _lib


def lib():
    return _load()


def _check(st: int):
    if st != 0:
        raise LowramError(st, _load().lowram_last_error().decode())


def _p(t: Optional[torch.Tensor]):
    return None if t is None else _vp(t.data_ptr())


def _stream():
    return _vp(torch.cuda.current_stream().cuda_stream)


def _act(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LOWRAM_F32
    if t.dtype == torch.bfloat16:
        return LOWRAM_BF16
    raise TypeError(f"activation dtype {t.dtype} (float32 or bfloat16)")


def _dev(*ts):
    """Every tensor given is a contiguous CUDA tensor, and all of them live on one device, which is returned.  The
    C entry points launch on the current device and stream, so each wrapper makes that device current for its call
    (`_on`); a pointer of another GPU would be read by this device's kernels."""
    dev = None
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("tensors must be contiguous CUDA tensors")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise LowramShapeError(f"tensors on {dev} and {t.device}: every tensor of a call must be on one device")
    return dev


def _on(dev):
    """Make `dev` the current CUDA device for the library call (its stream, launches and device queries)."""
    return torch.cuda.device(dev)


def _workspace(nbytes: int, workspace: Optional[torch.Tensor], device) -> torch.Tensor:
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError(f"workspace too small: {nbytes} bytes needed")
        return workspace
    return torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------------------------------------
# RoPE tables
# ------------------------------------------------------------------------------------------------
def lowram_rope_table(d: int, theta: float, max_pos: int, device="cuda"):
    """cos/sin tables [d/2, max_pos] float32 (frequency-major) built on the device in fp64."""
    cos = torch.empty((d // 2, max_pos), dtype=torch.float32, device=device)
    sin = torch.empty_like(cos)
    with _on(_dev(cos, sin)):
        _check(_load().lowram_rope_table(int(d), float(theta), int(max_pos), _p(cos), _p(sin), _stream()))
    return cos, sin


# ------------------------------------------------------------------------------------------------
# decode
# ------------------------------------------------------------------------------------------------
def decode_shape(q, coef, w1, *, S: int, n_res: int, max_pos: int, res_dtype: int, sm_scale: float = 0.0,
                 coef_int4: bool = False, basis=None, int4_exact_split: bool = False) -> lowram_decode_shape:
    """The C shape of a decode call.  A basis [B, H_kv*d, r] (one per sequence) or a w1 [B, H_kv, m, d] (a predictor
    per sequence) sets the matching batch stride to one sequence's elements; [H_kv*d, r] / [H_kv, m, d] share
    them across the batch (stride 0)."""
    B, H_q, d = q.shape
    T = coef.shape[1]
    r = coef.shape[2] * 2 if coef_int4 else coef.shape[2]
    per_seq_mlp = w1.dim() == 4
    H_kv, m = (w1.shape[1], w1.shape[2]) if per_seq_mlp else (w1.shape[0], w1.shape[1])
    act = _act(q)
    sh = lowram_decode_shape(B, T, H_q, H_kv, d, r, m, int(S), int(n_res), act,
                             LOWRAM_INT4_G32 if coef_int4 else _act(coef), int(res_dtype), int(max_pos),
                             float(sm_scale))
    if basis is not None and basis.dim() == 3:
        sh.basis_batch_stride = basis[0].numel()
    if per_seq_mlp:
        sh.mlp_batch_stride = w1[0].numel()
    if int4_exact_split:
        sh.flags |= FLAG_INT4_EXACT_SPLIT
    return sh


def _check_decode_buffers(s: lowram_decode_shape, *, q, coef, coef_scale, pos, rope_cos, rope_sin, basis, w1, w2,
                          b1, b2, res_idx, res_val, res_scale, out, lse, sel_out=None, key_out=None):
    B, T, H_q, H_kv, d, r, m = s.B, s.T, s.H_q, s.H_kv, s.d, s.r, s.m
    act = _ESZ[s.act_dtype]
    _need("q", q, B * H_q * d, act)
    if s.coef_dtype == LOWRAM_INT4_G32:
        _need("coef", coef, B * T * r // 2, 1)
        if coef_scale is None:
            raise LowramShapeError("coef_scale is required for int4 coefficients")
        _need("coef_scale", coef_scale, B * T * r // 32, 2)
    else:
        _need("coef", coef, B * T * r, _ESZ[s.coef_dtype])
    _need("pos", pos, B * T, 4)
    _need("rope_cos", rope_cos, d // 2 * s.max_pos, 4)
    _need("rope_sin", rope_sin, d // 2 * s.max_pos, 4)
    sb, sm = s.basis_batch_stride, s.mlp_batch_stride
    nb = (B - 1) * sb + H_kv * d * r if (sb and B) else H_kv * d * r
    nm = (B - 1) * sm + H_kv * m * d if (sm and B) else H_kv * m * d
    _need("basis", basis, nb, act)
    _need("w1", w1, nm, act)
    _need("w2", w2, nm, act)
    _need("b1", b1, (B if sm else 1) * H_kv * m, 4)
    _need("b2", b2, (B if sm else 1) * H_kv * d, 4)
    _need("res_idx", res_idx, B * H_kv * s.n_res, 4)
    _need("res_val", res_val, B * H_kv * s.n_res * d, 1 if s.res_dtype == LOWRAM_INT8_VEC else _ESZ[s.res_dtype])
    _need("res_scale", res_scale, B * H_kv * s.n_res, 2)
    _need("out", out, B * H_q * d, 4)
    _need("lse", lse, B * H_q, 4)
    _need("sel_out", sel_out, B * H_kv * min(s.S, T), 4)
    _need("key_out", key_out, B * H_kv * T, 4)


def lowram_decode_uses_tensor_cores(shape: lowram_decode_shape) -> bool:
    y = ctypes.c_int32(0)
    _check(_load().lowram_decode_uses_tensor_cores(ctypes.byref(shape), ctypes.byref(y)))
    return bool(y.value)


def lowram_decode_workspace_size(shape: lowram_decode_shape) -> int:
    n = ctypes.c_size_t(0)
    _check(_load().lowram_decode_workspace_size(ctypes.byref(shape), ctypes.byref(n)))
    return int(n.value)


def lowram_decode_attn(q: torch.Tensor, coef: torch.Tensor, basis: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor,
                       *, rope_cos: torch.Tensor, rope_sin: torch.Tensor, S: int,
                       coef_scale: Optional[torch.Tensor] = None, pos: Optional[torch.Tensor] = None,
                       b1: Optional[torch.Tensor] = None, b2: Optional[torch.Tensor] = None,
                       res_idx: Optional[torch.Tensor] = None, res_val: Optional[torch.Tensor] = None,
                       res_scale: Optional[torch.Tensor] = None, sm_scale: float = 0.0,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       sel_out: Optional[torch.Tensor] = None, key_out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, want_lse: bool = True, events=None,
                       int4_exact_split: bool = False):
    """Decode-step attention of one layer read from the compressed cache.  Returns (out, lse).

    int4_exact_split: int4 coefficients reach the tensor cores as an exact two-term bf16 split (rank 2r) instead of
    the default fp16 copy (LOWRAM_FLAG_INT4_EXACT_SPLIT).

    events: optional sequence of five recorded torch.cuda.Event objects (timing marks between the kernels,
    see lowram_decode_attn_events).

    Layouts as in include/lowram.h: q [B,H_q,d]; coef [B,T,r] (uint8 [B,T,r/2] + coef_scale fp16 [B,T,r/32] for
    int4); basis [H_kv*d, r], or [B, H_kv*d, r] for a basis per sequence; w1 [H_kv,m,d] and w2 [H_kv,d,m], or
    [B,H_kv,m,d] and [B,H_kv,d,m] (with b1 [B,H_kv,m], b2 [B,H_kv,d]) for a predictor per sequence;
    res_idx int32 [B,H_kv,n_res]; res_val [B,H_kv,n_res,d] (int8 + res_scale fp16 [B,H_kv,n_res] for the int8
    format); rope tables [d/2, max_pos].
    """
    coef_int4 = coef.dtype == torch.uint8
    n_res = 0 if res_idx is None else int(res_idx.shape[-1])
    if res_val is None:
        res_dtype = _act(q)
    elif res_val.dtype == torch.int8:
        res_dtype = LOWRAM_INT8_VEC
    else:
        res_dtype = _act(res_val)
    shape = decode_shape(q, coef, w1, S=S, n_res=n_res, max_pos=rope_cos.shape[1], res_dtype=res_dtype,
                         sm_scale=sm_scale, coef_int4=coef_int4, basis=basis, int4_exact_split=int4_exact_split)
    _check_decode_buffers(shape, q=q, coef=coef, coef_scale=coef_scale, pos=pos, rope_cos=rope_cos, rope_sin=rope_sin,
                          basis=basis, w1=w1, w2=w2, b1=b1, b2=b2, res_idx=res_idx, res_val=res_val,
                          res_scale=res_scale, out=out, lse=lse, sel_out=sel_out, key_out=key_out)
    dev = _dev(q, coef, basis, w1, w2, rope_cos, rope_sin, coef_scale, pos, b1, b2, res_idx, res_val, res_scale,
               out, lse, sel_out, key_out, workspace)
    B, H_q, d = q.shape
    if out is None:
        out = torch.empty((B, H_q, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    ws = _workspace(lowram_decode_workspace_size(shape), workspace, dev)
    with _on(dev):
        args = (ctypes.byref(shape), _p(q), _p(coef), _p(coef_scale), _p(pos), _p(rope_cos), _p(rope_sin), _p(basis),
                _p(w1), _p(w2), _p(b1), _p(b2), _p(res_idx), _p(res_val), _p(res_scale), _p(out), _p(lse),
                _p(sel_out), _p(key_out), _p(ws), ws.numel() * ws.element_size(), _stream())
        if events is None:
            _check(_load().lowram_decode_attn(*args))
        else:
            arr = (ctypes.c_void_p * 5)(*[None if e is None else e.cuda_event for e in events])
            _check(_load().lowram_decode_attn_events(*args, ctypes.cast(arr, _vp)))
    return out, lse


def lowram_decode_attn_static(q: torch.Tensor, coef: torch.Tensor, basis: torch.Tensor, w1: torch.Tensor,
                              w2: torch.Tensor, *, rope_cos: torch.Tensor, rope_sin: torch.Tensor, S: int,
                              out: torch.Tensor, lse: Optional[torch.Tensor] = None,
                              coef_scale: Optional[torch.Tensor] = None, pos: Optional[torch.Tensor] = None,
                              b1: Optional[torch.Tensor] = None, b2: Optional[torch.Tensor] = None,
                              res_idx: Optional[torch.Tensor] = None, res_val: Optional[torch.Tensor] = None,
                              res_scale: Optional[torch.Tensor] = None, sm_scale: float = 0.0):
    """lowram_decode_attn for callers that cannot allocate: the library's static device scratch replaces the
    workspace (see include/lowram.h).  The caller passes every input and preallocated outputs; this wrapper
    allocates nothing."""
    coef_int4 = coef.dtype == torch.uint8
    n_res = 0 if res_idx is None else int(res_idx.shape[-1])
    if res_val is None:
        res_dtype = _act(q)
    elif res_val.dtype == torch.int8:
        res_dtype = LOWRAM_INT8_VEC
    else:
        res_dtype = _act(res_val)
    shape = decode_shape(q, coef, w1, S=S, n_res=n_res, max_pos=rope_cos.shape[1], res_dtype=res_dtype,
                         sm_scale=sm_scale, coef_int4=coef_int4, basis=basis)
    if out is None:
        raise LowramShapeError("out is required (this call allocates nothing)")
    _check_decode_buffers(shape, q=q, coef=coef, coef_scale=coef_scale, pos=pos, rope_cos=rope_cos, rope_sin=rope_sin,
                          basis=basis, w1=w1, w2=w2, b1=b1, b2=b2, res_idx=res_idx, res_val=res_val,
                          res_scale=res_scale, out=out, lse=lse)
    dev = _dev(q, coef, basis, w1, w2, rope_cos, rope_sin, coef_scale, pos, b1, b2, res_idx, res_val, res_scale,
               out, lse)
    with _on(dev):
        _check(_load().lowram_decode_attn_static(ctypes.byref(shape), _p(q), _p(coef), _p(coef_scale), _p(pos),
                                                 _p(rope_cos), _p(rope_sin), _p(basis), _p(w1), _p(w2), _p(b1),
                                                 _p(b2), _p(res_idx), _p(res_val), _p(res_scale), _p(out), _p(lse),
                                                 None, None, _stream()))
    return out, lse


def lowram_decode_attn_static_get_error(device=None) -> int:
    """Device check word of the static scratch of `device` (default: the current device), cleared afterwards.
    Synchronises the current stream of that device."""
    w = ctypes.c_uint32(0)
    with _on(torch.cuda.current_device() if device is None else device):
        st = _load().lowram_decode_attn_static_get_error(_stream(), ctypes.byref(w))
    if st not in (0, 6):
        _check(st)
    return int(w.value)


# ------------------------------------------------------------------------------------------------
# compress
# ------------------------------------------------------------------------------------------------
def _ptr_array(ts: Optional[Sequence[Optional[torch.Tensor]]]):
    if ts is None:
        return None
    arr = (ctypes.c_void_p * len(ts))(*[None if t is None else t.data_ptr() for t in ts])
    return arr


def lowram_compress_workspace_size(shape: lowram_compress_shape) -> int:
    n = ctypes.c_size_t(0)
    _check(_load().lowram_compress_workspace_size(ctypes.byref(shape), ctypes.byref(n)))
    return int(n.value)


def lowram_compress(keys: torch.Tensor, values: Sequence[torch.Tensor], proj: torch.Tensor,
                    bases: Sequence[torch.Tensor], w1s: Sequence[torch.Tensor], w2s: Sequence[torch.Tensor], *,
                    n_res: int, coef_dtype: int, res_dtype: int, pos: Optional[torch.Tensor] = None,
                    rope_cos: Optional[torch.Tensor] = None, rope_sin: Optional[torch.Tensor] = None,
                    keys_post_rope: bool = False, b1s=None, b2s=None, want_err: bool = False,
                    workspace: Optional[torch.Tensor] = None) -> dict:
    """Write side of one layer group.  keys [B,T,G,H_kv,d]; values G x [B,T,H_kv,d]; proj [r, G*H_kv*d] float32."""
    B, T, G, H_kv, d = keys.shape
    r = proj.shape[0]
    m = w1s[0].shape[1]
    dev = keys.device
    shape = lowram_compress_shape(B, T, G, H_kv, d, r, m, int(n_res), _act(keys), int(coef_dtype), int(res_dtype),
                                  int(bool(keys_post_rope)), 0 if rope_cos is None else rope_cos.shape[1])
    act = _ESZ[_act(keys)]
    D = G * H_kv * d
    _need_list("values", values, G, B * T * H_kv * d, act)
    _need("proj", proj, r * D, 4)
    _need("pos", pos, B * T, 4)
    _need("rope_cos", rope_cos, d // 2 * shape.max_pos, 4)
    _need("rope_sin", rope_sin, d // 2 * shape.max_pos, 4)
    _need_list("bases", bases, G, H_kv * d * r, act)
    _need_list("w1s", w1s, G, H_kv * m * d, act)
    _need_list("w2s", w2s, G, H_kv * d * m, act)
    _need_list("b1s", b1s, G, H_kv * m, 4)
    _need_list("b2s", b2s, G, H_kv * d, 4)
    dev = _dev(keys, proj, pos, rope_cos, rope_sin, workspace, *values, *bases, *w1s, *w2s, *(b1s or []),
               *(b2s or []))
    if coef_dtype == LOWRAM_INT4_G32:
        coef = torch.empty((B, T, r // 2), dtype=torch.uint8, device=dev)
        coef_scale = torch.empty((B, T, r // 32), dtype=torch.float16, device=dev)
    else:
        coef = torch.empty((B, T, r), dtype=torch.float32 if coef_dtype == LOWRAM_F32 else torch.bfloat16, device=dev)
        coef_scale = None
    res_idx = [torch.empty((B, H_kv, n_res), dtype=torch.int32, device=dev) for _ in range(G)]
    if res_dtype == LOWRAM_INT8_VEC:
        res_val = [torch.empty((B, H_kv, n_res, d), dtype=torch.int8, device=dev) for _ in range(G)]
        res_scale = [torch.empty((B, H_kv, n_res), dtype=torch.float16, device=dev) for _ in range(G)]
    else:
        vdt = torch.float32 if res_dtype == LOWRAM_F32 else torch.bfloat16
        res_val = [torch.empty((B, H_kv, n_res, d), dtype=vdt, device=dev) for _ in range(G)]
        res_scale = None
    err = [torch.empty((B, H_kv, T), dtype=torch.float32, device=dev) for _ in range(G)] if want_err else None
    ws = _workspace(lowram_compress_workspace_size(shape), workspace, dev)
    arrays = {name: _ptr_array(ts) for name, ts in (("values", values), ("basis", bases), ("w1", w1s), ("w2", w2s),
                                                   ("b1", b1s), ("b2", b2s), ("res_idx", res_idx),
                                                   ("res_val", res_val), ("res_scale", res_scale), ("err", err))}
    ap = {k: (None if v is None else ctypes.cast(v, _vp)) for k, v in arrays.items()}
    with _on(dev):
        _check(_load().lowram_compress(ctypes.byref(shape), _p(keys), ap["values"], _p(proj), _p(pos), _p(rope_cos),
                                       _p(rope_sin), ap["basis"], ap["w1"], ap["w2"], ap["b1"], ap["b2"], _p(coef),
                                       _p(coef_scale), ap["res_idx"], ap["res_val"], ap["res_scale"], ap["err"],
                                       _p(ws), ws.numel() * ws.element_size(), _stream()))
    return {"coef": coef, "coef_scale": coef_scale, "res_idx": res_idx, "res_val": res_val, "res_scale": res_scale,
            "err": err, "workspace": ws}


# ------------------------------------------------------------------------------------------------
# dense comparator
# ------------------------------------------------------------------------------------------------
def lowram_dense_workspace_size(B: int, T: int, H_q: int, H_kv: int, d: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_load().lowram_dense_workspace_size(B, T, H_q, H_kv, d, ctypes.byref(n)))
    return int(n.value)


def lowram_dense_decode_attn(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, sm_scale: float = 0.0,
                             out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                             workspace: Optional[torch.Tensor] = None, want_lse: bool = True):
    """Plain decode attention over explicit rotated K and V [B,T,H_kv,d]; q [B,H_q,d].  Returns (out, lse)."""
    B, H_q, d = q.shape
    T, H_kv = k.shape[1], k.shape[2]
    act = _ESZ[_act(q)]
    _need("k", k, B * T * H_kv * d, act)
    _need("v", v, B * T * H_kv * d, act)
    _need("out", out, B * H_q * d, 4)
    _need("lse", lse, B * H_q, 4)
    dev = _dev(q, k, v, out, lse, workspace)
    if out is None:
        out = torch.empty((B, H_q, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    ws = _workspace(lowram_dense_workspace_size(B, T, H_q, H_kv, d), workspace, dev)
    with _on(dev):
        _check(_load().lowram_dense_decode_attn(B, T, H_q, H_kv, d, _act(q), float(sm_scale), _p(q), _p(k), _p(v),
                                                _p(out), _p(lse), _p(ws), ws.numel() * ws.element_size(), _stream()))
    return out, lse


# ------------------------------------------------------------------------------------------------
# heavy hitters from accumulated attention: the tokens an evicted cache keeps
# ------------------------------------------------------------------------------------------------
def lowram_attention_mass_workspace_size(B: int, T: int, W: int, H_q: int, H_kv: int, d: int, dtype: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_load().lowram_attention_mass_workspace_size(B, T, W, H_q, H_kv, d, int(dtype), ctypes.byref(n)))
    return int(n.value)


def lowram_evict_plan_workspace_size(B: int, T: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_load().lowram_evict_plan_workspace_size(B, T, ctypes.byref(n)))
    return int(n.value)


def lowram_attention_mass(q_win: torch.Tensor, k: torch.Tensor, *, sm_scale: float = 0.0,
                          workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Attention mass [B, T] of every prompt token from the window queries q_win [B, W, H_q, d] (k [B, T, H_kv, d])."""
    B, W, H_q, d = q_win.shape
    T, H_kv = k.shape[1], k.shape[2]
    if q_win.dtype != k.dtype:
        raise TypeError("q_win and k must share one dtype")
    _need("k", k, B * T * H_kv * d, _ESZ[_act(k)])
    dev = _dev(q_win, k, workspace)
    ws = _workspace(lowram_attention_mass_workspace_size(B, T, W, H_q, H_kv, d, _act(k)), workspace, dev)
    mass = torch.empty((B, T), dtype=torch.float32, device=dev)
    with _on(dev):
        _check(_load().lowram_attention_mass(B, T, W, H_q, H_kv, d, _act(k), float(sm_scale), _p(q_win), _p(k),
                                             _p(mass), _p(ws), ws.numel() * ws.element_size(), _stream()))
    return mass


def lowram_evict_plan(mass: torch.Tensor, *, n_sink: int, n_recent: int, T_keep: int,
                      workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Kept token indices [B, T_keep] (ascending): sinks, recents and the heaviest others by mass [B, T]."""
    B, T = mass.shape
    dev = _dev(mass, workspace)
    ws = _workspace(lowram_evict_plan_workspace_size(B, T), workspace, dev)
    keep = torch.empty((B, int(T_keep)), dtype=torch.int32, device=dev)
    with _on(dev):
        _check(_load().lowram_evict_plan(B, T, int(n_sink), int(n_recent), int(T_keep), _p(mass), _p(keep), _p(ws),
                                         ws.numel() * ws.element_size(), _stream()))
    return keep


# ------------------------------------------------------------------------------------------------
# test-time fit of the value predictor (float32 master parameters, updated in place)
# ------------------------------------------------------------------------------------------------
def _pred_dims(keys, values, w1, w2):
    B, T, H_kv, d = keys.shape
    m = w1.shape[1]
    _dev(keys, values, w1, w2)
    if values.shape != keys.shape or values.dtype != keys.dtype:
        raise ValueError("keys and values must share shape [B, T, H_kv, d] and dtype")
    if w1.shape != (H_kv, m, d) or w2.shape != (H_kv, d, m):
        raise ValueError("w1 [H_kv, m, d] and w2 [H_kv, d, m] expected")
    return B, T, H_kv, d, m


def _pred_params(H_kv, d, m, w1, b1, w2, b2):
    for t in (w1, b1, w2, b2):
        if t.dtype != torch.float32:
            raise TypeError("predictor parameters are float32")
    _need("b1", b1, H_kv * m, 4)
    _need("b2", b2, H_kv * d, 4)


def lowram_predictor_grad(keys: torch.Tensor, values: torch.Tensor, w1: torch.Tensor, b1: torch.Tensor,
                          w2: torch.Tensor, b2: torch.Tensor):
    """Loss [H_kv] and gradient (g_w1, g_b1, g_w2, g_b2) of every head's predictor; parameters float32."""
    B, T, H_kv, d, m = _pred_dims(keys, values, w1, w2)
    _pred_params(H_kv, d, m, w1, b1, w2, b2)
    dev = _dev(keys, values, w1, b1, w2, b2)
    loss = torch.empty(H_kv, dtype=torch.float32, device=dev)
    g = [torch.empty_like(t) for t in (w1, b1, w2, b2)]
    with _on(dev):
        _check(_load().lowram_predictor_grad(B, T, H_kv, d, m, _act(keys), _p(keys), _p(values), _p(w1), _p(b1),
                                             _p(w2), _p(b2), _p(loss), *[_p(x) for x in g], _stream()))
    return (loss, *g)


def lowram_fit_predictor(keys: torch.Tensor, values: torch.Tensor, w1: torch.Tensor, b1: torch.Tensor,
                         w2: torch.Tensor, b2: torch.Tensor, *, steps: int, lr: float, beta1: float = 0.9,
                         beta2: float = 0.999, eps: float = 1e-8, want_losses: bool = True,
                         workspace: Optional[torch.Tensor] = None):
    """`steps` full-batch Adam steps on every head's predictor, parameters (float32) updated in place.
    Returns the losses [steps, H_kv] before each step (or None)."""
    B, T, H_kv, d, m = _pred_dims(keys, values, w1, w2)
    _pred_params(H_kv, d, m, w1, b1, w2, b2)
    dev = _dev(keys, values, w1, b1, w2, b2, workspace)
    n = ctypes.c_size_t(0)
    _check(_load().lowram_fit_predictor_workspace_size(B, T, H_kv, d, m, ctypes.byref(n)))
    ws = _workspace(n.value, workspace, dev)
    losses = torch.empty((int(steps), H_kv), dtype=torch.float32, device=dev) if want_losses else None
    with _on(dev):
        _check(_load().lowram_fit_predictor(B, T, H_kv, d, m, _act(keys), _p(keys), _p(values), int(steps), float(lr),
                                            float(beta1), float(beta2), float(eps), _p(w1), _p(b1), _p(w2), _p(b2),
                                            _p(losses), _p(ws), ws.numel() * ws.element_size(), _stream()))
    return losses


# ------------------------------------------------------------------------------------------------
# fitted basis: cross-layer SVD of the RoPE-inverted keys (the proj and bases lowram_compress takes)
# ------------------------------------------------------------------------------------------------
def lowram_fit_basis(keys: torch.Tensor, r: int, *, pos: Optional[torch.Tensor] = None,
                     rope_cos: Optional[torch.Tensor] = None, rope_sin: Optional[torch.Tensor] = None,
                     keys_post_rope: bool = False, iters: int = 8, seed: int = 0,
                     workspace: Optional[torch.Tensor] = None):
    """keys [B, T, G, H_kv, d] -> (proj [r, G*H_kv*d] float32, bases G x [H_kv*d, r] in keys' dtype, workspace)."""
    B, T, G, H_kv, d = keys.shape
    dev = keys.device
    shape = lowram_compress_shape(B, T, G, H_kv, d, int(r), 32, 0, _act(keys), LOWRAM_BF16, LOWRAM_BF16,
                                  int(bool(keys_post_rope)), 0 if rope_cos is None else rope_cos.shape[1])
    _need("pos", pos, B * T, 4)
    _need("rope_cos", rope_cos, d // 2 * shape.max_pos, 4)
    _need("rope_sin", rope_sin, d // 2 * shape.max_pos, 4)
    dev = _dev(keys, pos, rope_cos, rope_sin, workspace)
    n = ctypes.c_size_t(0)
    _check(_load().lowram_fit_basis_workspace_size(ctypes.byref(shape), ctypes.byref(n)))
    ws = _workspace(n.value, workspace, dev)
    proj = torch.empty((int(r), G * H_kv * d), dtype=torch.float32, device=dev)
    bases = [torch.empty((H_kv * d, int(r)), dtype=keys.dtype, device=dev) for _ in range(G)]
    arr = _ptr_array(bases)
    with _on(dev):
        _check(_load().lowram_fit_basis(ctypes.byref(shape), _p(keys), _p(pos), _p(rope_cos), _p(rope_sin),
                                        int(iters), int(seed) & 0xFFFFFFFFFFFFFFFF, _p(proj), ctypes.cast(arr, _vp),
                                        _p(ws), ws.numel() * ws.element_size(), _stream()))
    return proj, bases, ws


# ------------------------------------------------------------------------------------------------
# exact tail: tokens decoded after compression, kept as explicit rotated K and V
# ------------------------------------------------------------------------------------------------
def lowram_tail_append(k_new: torch.Tensor, v_new: torch.Tensor, tail_k: torch.Tensor, tail_v: torch.Tensor, t: int):
    """Write one token's rotated keys and values [B, H_kv, d] into row t of the tail buffers [B, T_cap, H_kv, d]."""
    B, T_cap, H_kv, d = tail_k.shape
    dev = _dev(k_new, v_new, tail_k, tail_v)
    if k_new.shape != (B, H_kv, d) or v_new.shape != (B, H_kv, d) or tail_v.shape != tail_k.shape:
        raise ValueError("k_new, v_new must be [B, H_kv, d] and the tail buffers [B, T_cap, H_kv, d]")
    if not (k_new.dtype == v_new.dtype == tail_k.dtype == tail_v.dtype):
        raise TypeError("k_new, v_new and the tail buffers must share one dtype")
    with _on(dev):
        _check(_load().lowram_tail_append(B, T_cap, H_kv, d, _act(tail_k), int(t), _p(k_new), _p(v_new), _p(tail_k),
                                          _p(tail_v), _stream()))


def lowram_tail_decode_attn(q: torch.Tensor, tail_k: torch.Tensor, tail_v: torch.Tensor, t_len: int, *,
                            sm_scale: float = 0.0, out: Optional[torch.Tensor] = None,
                            lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                            want_lse: bool = True):
    """Attention of q [B, H_q, d] over the first t_len rows of the tail buffers, read in place.  Returns (out, lse)."""
    B, H_q, d = q.shape
    T_cap, H_kv = tail_k.shape[1], tail_k.shape[2]
    act = _ESZ[_act(q)]
    _need("tail_k", tail_k, B * T_cap * H_kv * d, act)
    _need("tail_v", tail_v, B * T_cap * H_kv * d, act)
    _need("out", out, B * H_q * d, 4)
    _need("lse", lse, B * H_q, 4)
    dev = _dev(q, tail_k, tail_v, out, lse, workspace)
    if out is None:
        out = torch.empty((B, H_q, d), dtype=torch.float32, device=dev)
    if lse is None and want_lse:
        lse = torch.empty((B, H_q), dtype=torch.float32, device=dev)
    ws = _workspace(lowram_dense_workspace_size(B, int(t_len), H_q, H_kv, d), workspace, dev)
    with _on(dev):
        _check(_load().lowram_tail_decode_attn(B, T_cap, int(t_len), H_q, H_kv, d, _act(q), float(sm_scale), _p(q),
                                               _p(tail_k), _p(tail_v), _p(out), _p(lse), _p(ws),
                                               ws.numel() * ws.element_size(), _stream()))
    return out, lse


def lowram_merge_attn(out_a: torch.Tensor, lse_a: torch.Tensor, out_b: torch.Tensor, lse_b: torch.Tensor, *,
                      out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None):
    """Merge two attention results over disjoint token sets through their log-sum-exp.  Returns (out, lse);
    out / lse may be given as out_a / lse_a for an in-place merge."""
    B, H_q, d = out_a.shape
    for t in (out_a, lse_a, out_b, lse_b):
        if t.dtype != torch.float32:
            raise TypeError("merge operands are float32")
    _need("lse_a", lse_a, B * H_q, 4)
    _need("out_b", out_b, B * H_q * d, 4)
    _need("lse_b", lse_b, B * H_q, 4)
    _need("out", out, B * H_q * d, 4)
    _need("lse", lse, B * H_q, 4)
    dev = _dev(out_a, lse_a, out_b, lse_b, out, lse)
    if out is None:
        out = torch.empty_like(out_a)
    if lse is None:
        lse = torch.empty_like(lse_a)
    with _on(dev):
        _check(_load().lowram_merge_attn(B, H_q, d, _p(out_a), _p(lse_a), _p(out_b), _p(lse_b), _p(out), _p(lse),
                                         _stream()))
    return out, lse


# ------------------------------------------------------------------------------------------------
# status
# ------------------------------------------------------------------------------------------------
def lowram_get_error(workspace: torch.Tensor) -> int:
    """Device check word of a workspace (LOWRAM_CHECK_* bits), cleared afterwards.  Synchronises the stream."""
    w = ctypes.c_uint32(0)
    with _on(_dev(workspace)):
        st = _load().lowram_get_error(_p(workspace), _stream(), ctypes.byref(w))
    if st not in (0, 6):
        _check(st)
    return int(w.value)


def lowram_clear_error(workspace: torch.Tensor):
    with _on(_dev(workspace)):
        _check(_load().lowram_clear_error(_p(workspace), _stream()))


def lowram_version() -> int:
    return int(_load().lowram_version())


def lowram_set_wait_limit(cycles: int):
    """Testing aid: pipeline waits of the tensor-core value pass give up after `cycles` SM cycles (0: the default,
    about a second).  A call whose wait gives up sets CHECK_TIMEOUT in its workspace's check word."""
    _check(_load().lowram_set_wait_limit(int(cycles)))

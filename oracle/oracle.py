"""ctypes front end of the fp64 oracle (``lowram_oracle.c``) -- TEST INFRASTRUCTURE ONLY.

Every array is converted to fp64 exactly (bf16, fp16 and fp32 values are all representable in
double) before it reaches the C code.  Stored quantised formats are decoded by the oracle's own
dequantisers.  The functions below follow the method's steps in order; the docstrings name the web
page (by title and section) each step comes from.

Pages cited:
  [ABS] "LowRAM: Low-Rank Keys and Amortised Values for Composable KV Cache Compression at
        Test-Time" (arXiv listing), Abstract.
  [EX]  "LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression", sections "Value
        cache amortisation in plain language", "Asymmetric key compression with xKV",
        "Step-by-step mental model for one decoding session".
  [CB]  "LowRAM: predict values from keys, store only the misses", flowchart and Key points.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lowram_oracle.c")
_SO = os.path.join(_HERE, "liblowram_oracle.so")

__all__ = [
    "build", "lib", "Dims", "f64", "round_bf16", "round_f16", "round_f32", "quant_int4_g32",
    "dequant_int4_g32", "quant_int8_vec", "dequant_int8_vec", "rope", "rope_rows", "rope_angles", "mlp",
    "rebuild_keys", "predict_values", "decode", "project", "residuals", "compress_group",
    "dense_decode", "merge_attn", "fit_basis", "predictor_loss_grad", "adam_step", "fit_predictor",
    "attention_mass", "evict_plan", "top_n", "n_res_for", "max_threads", "store",
]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math) into ``liblowram_oracle.so``."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("B", "T", "H_q", "H_kv", "d", "r", "m", "S", "n_res")] + [
        ("rope_theta", ctypes.c_double), ("sm_scale", ctypes.c_double)]


_lib = None
_D = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.POINTER(ctypes.c_int32)
_U8 = ctypes.POINTER(ctypes.c_uint8)
_I8 = ctypes.POINTER(ctypes.c_int8)


def lib():
    """The compiled oracle.  LOWRAM_ORACLE_LIB may name another build of the same source (the mutation
    test points it at copies with planted mistakes)."""
    global _lib
    if _lib is None:
        L = ctypes.CDLL(os.environ.get("LOWRAM_ORACLE_LIB") or build())
        i64, ci, cd = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        sig = {
            "lro_round_bf16": (None, [i64, _D, _D]),
            "lro_round_f32": (None, [i64, _D, _D]),
            "lro_round_f16_scalar": (cd, [cd]),
            "lro_quant_int4_g32": (None, [i64, ci, _D, _U8, _D]),
            "lro_dequant_int4_g32": (None, [i64, ci, _U8, _D, _D]),
            "lro_quant_int8_vec": (None, [i64, ci, _D, _I8, _D]),
            "lro_dequant_int8_vec": (None, [i64, ci, _I8, _D, _D]),
            "lro_rope_angles": (None, [ci, cd, cd, _D, _D]),
            "lro_rope": (None, [ci, cd, cd, _D, _D, ci]),
            "lro_rope_rows": (None, [i64, ci, cd, _I32, _D, _D, ci]),
            "lro_mlp": (None, [ci, ci, _D, _D, _D, _D, _D, _D, _D]),
            "lro_top_n": (None, [ci, _D, ci, _I32]),
            "lro_decode": (ci, [ctypes.POINTER(Dims), _D, _D, _I32, _D, _D, _D, _D, _D, _I32, _D,
                                _D, _D, _D, _I32, ci]),
            "lro_project": (ci, [ci, ci, ci, ci, ci, ci, _D, _I32, ci, cd, _D, _D, ci]),
            "lro_residuals": (ci, [ctypes.POINTER(Dims), _D, _D, _D, _D, _D, _D, _D, _I32, _D, _D, ci]),
            "lro_dense_decode": (ci, [ci, ci, ci, ci, ci, cd, _D, _D, _D, _D, _D, ci]),
            "lro_rebuild_keys": (ci, [ctypes.POINTER(Dims), _D, _D, _D, ci]),
            "lro_predict_values": (ci, [ci, ci, ci, ci, ci, _D, _D, _D, _D, _D, _D, ci]),
            "lro_max_threads": (ci, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


# ---------------------------------------------------------------------------------------------
# array plumbing
# ---------------------------------------------------------------------------------------------
def f64(x) -> np.ndarray:
    """Exact conversion of a torch tensor or array-like to a contiguous float64 numpy array."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.int32).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _p(a, ty=_D):
    return None if a is None else a.ctypes.data_as(ty)


def _chk(status: int, what: str):
    if status != 0:
        raise RuntimeError(f"oracle {what} failed with status {status}")


def max_threads() -> int:
    return int(lib().lro_max_threads())


# ---------------------------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round to bfloat16 (nearest, ties to even), returned as exactly representable fp64 values."""
    a = f64(x)
    y = np.empty_like(a)
    lib().lro_round_bf16(a.size, _p(a), _p(y))
    return y


def round_f32(x) -> np.ndarray:
    a = f64(x)
    y = np.empty_like(a)
    lib().lro_round_f32(a.size, _p(a), _p(y))
    return y


def round_f16(x) -> np.ndarray:
    a = f64(x)
    return np.vectorize(lib().lro_round_f16_scalar, otypes=[np.float64])(a) if a.size else a.copy()


def quant_int4_g32(x):
    """int4 codes in groups of 32 with an fp16 scale -> (packed uint8 [..., r/2], scales fp64 [..., r/32])."""
    a = f64(x)
    r = a.shape[-1]
    rows = a.size // r
    packed = np.empty(a.shape[:-1] + (r // 2,), dtype=np.uint8)
    scales = np.empty(a.shape[:-1] + (r // 32,), dtype=np.float64)
    lib().lro_quant_int4_g32(rows, r, _p(a), _p(packed, _U8), _p(scales))
    return packed, scales


def dequant_int4_g32(packed, scales) -> np.ndarray:
    pk = np.ascontiguousarray(np.asarray(packed, dtype=np.uint8))
    sc = f64(scales)
    r = pk.shape[-1] * 2
    x = np.empty(pk.shape[:-1] + (r,), dtype=np.float64)
    lib().lro_dequant_int4_g32(pk.size // (r // 2), r, _p(pk, _U8), _p(sc), _p(x))
    return x


def quant_int8_vec(x):
    """int8 codes with one fp16 scale per last-axis vector -> (codes int8, scales fp64)."""
    a = f64(x)
    d = a.shape[-1]
    codes = np.empty(a.shape, dtype=np.int8)
    scales = np.empty(a.shape[:-1], dtype=np.float64)
    lib().lro_quant_int8_vec(a.size // d, d, _p(a), _p(codes, _I8), _p(scales))
    return codes, scales


def dequant_int8_vec(codes, scales) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.int8))
    sc = f64(scales)
    d = c.shape[-1]
    x = np.empty(c.shape, dtype=np.float64)
    lib().lro_dequant_int8_vec(c.size // d, d, _p(c, _I8), _p(sc), _p(x))
    return x


def store(x, fmt: str):
    """Round a fp64 tensor to a storage format: 'f64' (kept) | 'f32' | 'bf16' (values) or 'int4' | 'int8'
    (codes, scales)."""
    if fmt == "f64":
        return f64(x).copy()
    if fmt == "f32":
        return round_f32(x)
    if fmt == "bf16":
        return round_bf16(x)
    if fmt == "int4":
        return quant_int4_g32(x)
    if fmt == "int8":
        return quant_int8_vec(x)
    raise ValueError(fmt)


# ---------------------------------------------------------------------------------------------
# single steps
# ---------------------------------------------------------------------------------------------
def rope_angles(d: int, theta: float, pos: float):
    c = np.empty(d // 2)
    s = np.empty(d // 2)
    lib().lro_rope_angles(d, float(theta), float(pos), _p(c), _p(s))
    return c, s


def rope(x, pos: float, theta: float, inverse: bool = False) -> np.ndarray:
    """Rotate one d-vector at a position (rotate-half RoPE) [EX "Asymmetric key compression with xKV"]."""
    a = f64(x)
    y = np.empty_like(a)
    lib().lro_rope(a.shape[-1], float(theta), float(pos), _p(a), _p(y), int(bool(inverse)))
    return y


def rope_rows(x, pos, theta: float, inverse: bool = False) -> np.ndarray:
    """Rotate every d-vector of x [..., d]; pos has x's shape without the last axis (one position per vector)."""
    a = f64(x)
    d = a.shape[-1]
    P = np.ascontiguousarray(np.broadcast_to(_i32(pos), a.shape[:-1]), dtype=np.int32)
    y = np.empty_like(a)
    lib().lro_rope_rows(a.size // d, d, float(theta), _p(P, _I32), _p(a), _p(y), int(bool(inverse)))
    return y


def mlp(k_pre, w1, b1, w2, b2) -> np.ndarray:
    """One head's predictor on one pre-RoPE key: w2 . silu(w1 . k + b1) + b2 [ABS; EX "Value cache amortisation"]."""
    k, W1, W2 = f64(k_pre), f64(w1), f64(w2)
    B1, B2 = f64(b1), f64(b2)
    m, d = W1.shape
    hid = np.empty(m)
    v = np.empty(d)
    lib().lro_mlp(d, m, _p(W1), _p(B1), _p(W2), _p(B2), _p(k), _p(hid), _p(v))
    return v


def top_n(values, n: int) -> np.ndarray:
    """The n largest values (ties to the lower index), returned as ascending indices."""
    v = f64(values)
    out = np.empty(n, dtype=np.int32)
    lib().lro_top_n(v.size, _p(v), int(n), _p(out, _I32))
    return out


def _dims(B, T, H_q, H_kv, d, r, m, S, n_res, theta, sm_scale):
    return Dims(int(B), int(T), int(H_q), int(H_kv), int(d), int(r), int(m), int(S), int(n_res),
                float(theta), float(sm_scale))


def rebuild_keys(coef, basis, H_kv: int, d: int, threads: int = 0) -> np.ndarray:
    """Pre-RoPE keys [B, T, H_kv, d] of every token from coefficients [B, T, r] and basis [H_kv*d, r]."""
    C, W = f64(coef), f64(basis)
    B, T, r = C.shape
    out = np.empty((B, T, H_kv, d))
    D = _dims(B, T, H_kv, H_kv, d, r, 1, 0, 0, 1.0, 0.0)
    _chk(lib().lro_rebuild_keys(ctypes.byref(D), _p(C), _p(W), _p(out), threads), "rebuild_keys")
    return out


def predict_values(k_pre, w1, w2, b1=None, b2=None, threads: int = 0) -> np.ndarray:
    """Predicted values [B, T, H_kv, d] of every token from pre-RoPE keys [B, T, H_kv, d]."""
    K, W1, W2, B1, B2 = f64(k_pre), f64(w1), f64(w2), f64(b1), f64(b2)
    B, T, H_kv, d = K.shape
    m = W1.shape[1]
    out = np.empty_like(K)
    _chk(lib().lro_predict_values(B, T, H_kv, d, m, _p(K), _p(W1), _p(B1), _p(W2), _p(B2), _p(out), threads),
         "predict_values")
    return out


# ---------------------------------------------------------------------------------------------
# the two calls
# ---------------------------------------------------------------------------------------------
def n_res_for(rho: float, T: int) -> int:
    """Residual budget per (sequence, kv-head): the smallest count that keeps at least a fraction rho."""
    return max(0, min(T, int(math.ceil(rho * T - 1e-9))))


@dataclass
class DecodeResult:
    out: np.ndarray
    lse: np.ndarray
    key: np.ndarray
    sel: np.ndarray


def decode(q, coef, basis, w1, w2, *, S: int, theta: float, pos=None, b1=None, b2=None, res_idx=None,
           res_val=None, sm_scale: float = 0.0, threads: int = 0) -> DecodeResult:
    """One decode-step attention of one layer from the compressed cache (see ``lro_decode``).

    coef must already be decoded to values (``dequant_int4_g32`` for the int4 format); res_val likewise
    (``dequant_int8_vec``).  Shapes: q [B,H_q,d], coef [B,T,r], basis [H_kv*d,r], w1 [H_kv,m,d],
    w2 [H_kv,d,m], res_idx [B,H_kv,n_res], res_val [B,H_kv,n_res,d], pos [B,T] or None.

    A basis [B,H_kv*d,r] gives each sequence its own basis, and w1 [B,H_kv,m,d], w2 [B,H_kv,d,m] (with b1
    [B,H_kv,m], b2 [B,H_kv,d]) its own predictor: sequence b is then decoded with its own weights, one call
    per sequence (the sequences of a call share nothing else).
    """
    per_basis = np.ndim(basis) == 3
    per_mlp = np.ndim(w1) == 4
    if per_basis or per_mlp:
        parts = []
        for b in range(np.shape(q)[0]):
            pick = lambda x, on: None if x is None else (f64(x)[b] if on else x)
            sl = lambda x: None if x is None else f64(x)[b:b + 1]
            parts.append(decode(sl(q), sl(coef), pick(basis, per_basis), pick(w1, per_mlp), pick(w2, per_mlp), S=S,
                                theta=theta, pos=None if pos is None else _i32(pos)[b:b + 1],
                                b1=pick(b1, per_mlp), b2=pick(b2, per_mlp),
                                res_idx=None if res_idx is None else _i32(res_idx)[b:b + 1], res_val=sl(res_val),
                                sm_scale=sm_scale, threads=threads))
        return DecodeResult(*[np.concatenate([getattr(r, f) for r in parts]) for f in ("out", "lse", "key", "sel")])
    Q, C, W, W1, W2 = f64(q), f64(coef), f64(basis), f64(w1), f64(w2)
    B1, B2, RV = f64(b1), f64(b2), f64(res_val)
    RI, P = _i32(res_idx), _i32(pos)
    B, H_q, d = Q.shape
    T, r = C.shape[1], C.shape[2]
    H_kv, m = W1.shape[0], W1.shape[1]
    n_res = 0 if RI is None else RI.shape[-1]
    S_eff = min(S, T)
    out = np.empty((B, H_q, d))
    lse = np.empty((B, H_q))
    key = np.empty((B, H_kv, T))
    sel = np.empty((B, H_kv, S_eff), dtype=np.int32)
    D = _dims(B, T, H_q, H_kv, d, r, m, S, n_res, theta, sm_scale)
    _chk(lib().lro_decode(ctypes.byref(D), _p(Q), _p(C), _p(P, _I32), _p(W), _p(W1), _p(B1), _p(W2), _p(B2),
                          _p(RI, _I32), _p(RV), _p(out), _p(lse), _p(key), _p(sel, _I32), threads), "decode")
    return DecodeResult(out, lse, key, sel)


def project(k_cat, proj, G: int, H_kv: int, d: int, *, pos=None, keys_post_rope: bool = False,
            theta: float = 1e4, threads: int = 0) -> np.ndarray:
    """Latent coefficients [B, T, r] = proj . (RoPE-inverted) keys, unrounded [EX "Step-by-step", step 1]."""
    K, Pj, PS = f64(k_cat), f64(proj), _i32(pos)
    B, T = K.shape[0], K.shape[1]
    r = Pj.shape[0]
    K = K.reshape(B, T, G * H_kv * d)
    coef = np.empty((B, T, r))
    _chk(lib().lro_project(B, T, G, H_kv, d, r, _p(K), _p(PS, _I32), int(bool(keys_post_rope)), float(theta),
                           _p(Pj), _p(coef), threads), "project")
    return coef


def residuals(coef_stored, v, basis, w1, w2, n_res: int, *, b1=None, b2=None, threads: int = 0):
    """Worst-token residuals of one layer: (res_idx [B,H_kv,n_res], res_raw [B,H_kv,n_res,d], err [B,H_kv,T])."""
    C, V, W, W1, W2, B1, B2 = f64(coef_stored), f64(v), f64(basis), f64(w1), f64(w2), f64(b1), f64(b2)
    B, T, r = C.shape
    H_kv, d = V.shape[2], V.shape[3]
    m = W1.shape[1]
    ridx = np.empty((B, H_kv, n_res), dtype=np.int32)
    rraw = np.empty((B, H_kv, n_res, d))
    err = np.empty((B, H_kv, T))
    D = _dims(B, T, H_kv, H_kv, d, r, m, 0, n_res, 1.0, 0.0)
    _chk(lib().lro_residuals(ctypes.byref(D), _p(C), _p(V), _p(W), _p(W1), _p(B1), _p(W2), _p(B2),
                             _p(ridx, _I32), _p(rraw), _p(err), threads), "residuals")
    return ridx, rraw, err


def compress_group(k_cat, vs, proj, bases, w1s, w2s, *, G: int, H_kv: int, d: int, n_res: int,
                   coef_fmt: str = "bf16", res_fmt: str = "bf16", pos=None, keys_post_rope: bool = False,
                   theta: float = 1e4, b1s=None, b2s=None, threads: int = 0) -> dict:
    """The write side for one layer group, in the method's order [EX "Step-by-step mental model", step 1]:
    project the keys onto the latent coefficients and store them (rounded or quantised); then per layer
    rebuild the keys from the *stored* coefficients, predict values, rank tokens by error and keep the
    worst n_res as stored residuals [ABS; CB flowchart "Residual store: worst tokens only"].
    """
    coef_raw = project(k_cat, proj, G, H_kv, d, pos=pos, keys_post_rope=keys_post_rope, theta=theta,
                       threads=threads)
    res = {"coef_raw": coef_raw}
    if coef_fmt == "int4":
        packed, scales = quant_int4_g32(coef_raw)
        coef_vals = dequant_int4_g32(packed, scales)
        res.update(coef_q=packed, coef_scale=scales)
    else:
        coef_vals = store(coef_raw, coef_fmt)
    res["coef"] = coef_vals
    layers = []
    for li in range(G):
        ridx, rraw, err = residuals(coef_vals, vs[li], bases[li], w1s[li], w2s[li], n_res,
                                    b1=None if b1s is None else b1s[li], b2=None if b2s is None else b2s[li],
                                    threads=threads)
        entry = {"res_idx": ridx, "res_raw": rraw, "err": err}
        if res_fmt == "int8":
            codes, sc = quant_int8_vec(rraw)
            entry.update(res_q=codes, res_scale=sc, res_val=dequant_int8_vec(codes, sc))
        else:
            entry["res_val"] = store(rraw, res_fmt)
        layers.append(entry)
    res["layers"] = layers
    return res


def dense_decode(q, k, v, *, sm_scale: float = 0.0, threads: int = 0):
    """Plain softmax attention over explicit rotated keys and values [B, T, H_kv, d] -> (out, lse)."""
    Q, K, V = f64(q), f64(k), f64(v)
    B, H_q, d = Q.shape
    T, H_kv = K.shape[1], K.shape[2]
    out = np.empty((B, H_q, d))
    lse = np.empty((B, H_q))
    _chk(lib().lro_dense_decode(B, T, H_q, H_kv, d, float(sm_scale), _p(Q), _p(K), _p(V), _p(out), _p(lse),
                                threads), "dense_decode")
    return out, lse


def merge_attn(out_a, lse_a, out_b, lse_b):
    """Attention over the union of two disjoint token sets from the two sets' results: the tokens decoded after
    the prompt's cache was compressed stay explicit and are attended next to the compressed body [EX
    "Step-by-step mental model for one decoding session"].  With W = max(lse_a, lse_b), a = exp(lse_a - W),
    b = exp(lse_b - W): out = (a out_a + b out_b) / (a + b), lse = W + log(a + b); an empty set has lse = -inf
    (both empty: out = 0, lse = -inf).  Plain fp64 numpy."""
    oa, la, ob, lb = f64(out_a), f64(lse_a), f64(out_b), f64(lse_b)
    W = np.maximum(la, lb)
    empty = np.isneginf(W)
    Wf = np.where(empty, 0.0, W)
    a = np.where(empty, 0.0, np.exp(la - Wf))
    b = np.where(empty, 0.0, np.exp(lb - Wf))
    s = a + b
    with np.errstate(invalid="ignore", divide="ignore"):
        out = np.where(empty[..., None], 0.0, (a[..., None] * oa + b[..., None] * ob) / np.where(s == 0, 1.0, s)[..., None])
        lse = np.where(empty, -np.inf, Wf + np.log(np.where(s == 0, 1.0, s)))
    return out, lse


def fit_basis(k_cat, r: int, G: int, H_kv: int, d: int, *, pos=None, keys_post_rope: bool = False,
              theta: float = 1e4):
    """The group's shared low-rank key basis from the prompt's keys, the cross-layer SVD of the RoPE-inverted
    keys [EX "Asymmetric key compression with xKV": the G layers' keys are stacked and factored together, RoPE
    inverted first].  With k_cat [N = B*T, D = G*H_kv*d] (rotated back by each token's position when the keys
    are given rotated), the rank-r subspace of the largest singular values is spanned by the top-r eigenvectors
    U [D, r] of the Gram matrix k_cat^T k_cat (fp64, numpy.linalg.eigh as the eigensolver).
    Returns (proj [r, D] = U^T, bases [G] x [H_kv*d, r] = U's layer blocks, the r eigenvalues descending)."""
    K = f64(k_cat)
    B, T = K.shape[0], K.shape[1]
    K = K.reshape(B, T, G, H_kv, d)
    if keys_post_rope:
        P = np.arange(T)[None, :].repeat(B, 0) if pos is None else _i32(pos).astype(np.float64)
        K = rope_rows(K, np.broadcast_to(np.asarray(P)[:, :, None, None], (B, T, G, H_kv)), theta, inverse=True)
    K = K.reshape(B * T, G * H_kv * d)
    w, U = np.linalg.eigh(K.T @ K)
    order = np.argsort(w)[::-1][:r]
    U = U[:, order]
    return U.T.copy(), [U[l * H_kv * d:(l + 1) * H_kv * d].copy() for l in range(G)], w[order]


def predictor_loss_grad(k_pre, v, w1, b1, w2, b2):
    """Mean squared error of one kv-head's predictor over its tokens, and the gradient of that loss with respect
    to the predictor's parameters [ABS: the predictor is fitted at test time on the prompt; EX "Value cache
    amortisation in plain language": values are predicted from the pre-RoPE keys].  k_pre, v [N, d];
    w1 [m, d], b1 [m], w2 [d, m], b2 [d];  loss = 1/(N d) sum_t || w2 silu(w1 k_t + b1) + b2 - v_t ||^2.
    Plain fp64 numpy, the chain rule written out: silu'(z) = s + z s (1 - s) with s the logistic function.
    Returns (loss, g_w1, g_b1, g_w2, g_b2)."""
    K, V, W1, B1, W2, B2 = (f64(x) for x in (k_pre, v, w1, b1, w2, b2))
    N, d = K.shape
    Z = K @ W1.T + B1
    S = 1.0 / (1.0 + np.exp(-Z))
    H = Z * S
    E = H @ W2.T + B2 - V
    loss = float(np.sum(E * E) / (N * d))
    dV = 2.0 * E / (N * d)
    g_w2 = dV.T @ H
    g_b2 = dV.sum(axis=0)
    dZ = (dV @ W2) * (S + Z * S * (1.0 - S))
    g_w1 = dZ.T @ K
    g_b1 = dZ.sum(axis=0)
    return loss, g_w1, g_b1, g_w2, g_b2


def adam_step(p, g, m, v, step: int, lr: float, beta1: float, beta2: float, eps: float):
    """One Adam update (Kingma and Ba, with bias correction) of parameters p with gradient g; `step` counts from 1.
    Returns the new (p, m, v)."""
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    mh = m / (1.0 - beta1 ** step)
    vh = v / (1.0 - beta2 ** step)
    return p - lr * mh / (np.sqrt(vh) + eps), m, v


def fit_predictor(k_pre, v, w1, b1, w2, b2, *, steps: int, lr: float, beta1: float = 0.9, beta2: float = 0.999,
                  eps: float = 1e-8):
    """Test-time fit of every kv-head's predictor on the prompt's (pre-RoPE key, value) pairs: `steps` full-batch
    Adam steps on predictor_loss_grad from the given start.  k_pre, v [B, T, H_kv, d]; w1 [H_kv, m, d],
    b1 [H_kv, m], w2 [H_kv, d, m], b2 [H_kv, d].  Returns (w1, b1, w2, b2, losses [steps, H_kv]) where losses[s]
    is the loss before step s+1."""
    K, V = f64(k_pre), f64(v)
    B, T, H_kv, d = K.shape
    P = [f64(x).copy() for x in (w1, b1, w2, b2)]
    M = [np.zeros_like(x) for x in P]
    Vv = [np.zeros_like(x) for x in P]
    losses = np.zeros((steps, H_kv))
    for s in range(steps):
        for h in range(H_kv):
            Kh = K[:, :, h].reshape(B * T, d)
            Vh = V[:, :, h].reshape(B * T, d)
            loss, *g = predictor_loss_grad(Kh, Vh, P[0][h], P[1][h], P[2][h], P[3][h])
            losses[s, h] = loss
            for i in range(4):
                P[i][h], M[i][h], Vv[i][h] = adam_step(P[i][h], g[i], M[i][h], Vv[i][h], s + 1, lr, beta1, beta2, eps)
    return P[0], P[1], P[2], P[3], losses


def attention_mass(q_win, k, *, sm_scale: float = 0.0):
    """Attention mass each prompt token receives from an observation window of queries, for choosing the heavy
    hitters an evicted cache keeps [CB Key points / EX benchmarks: eviction keeps sinks, recent tokens and heavy
    hitters].  q_win [B, W, H_q, d] and k [B, T, H_kv, d] rotated; every window query attends all T tokens;
    mass[b, t] = sum_i sum_hq softmax_t(scale * q_win[b, i, hq] . k[b, t, hq // g])[t], g = H_q / H_kv.
    Plain fp64 numpy; the row sums are W * H_q."""
    Q, K = f64(q_win), f64(k)
    B, W, H_q, d = Q.shape
    T, H_kv = K.shape[1], K.shape[2]
    g = H_q // H_kv
    scale = sm_scale if sm_scale > 0 else d ** -0.5
    mass = np.zeros((B, T))
    for b in range(B):
        for hq in range(H_q):
            s = (Q[b, :, hq] @ K[b, :, hq // g].T) * scale            # [W, T]
            s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            mass[b] += (p / p.sum(axis=1, keepdims=True)).sum(axis=0)
    return mass


def evict_plan(mass, n_sink: int, n_recent: int, T_keep: int) -> np.ndarray:
    """Tokens an evicted cache keeps, per sequence, ascending: the first n_sink, the last n_recent, and the
    T_keep - n_sink - n_recent others of largest attention mass (ties to the lower index)."""
    M = f64(mass)
    B, T = M.shape
    keep = np.empty((B, T_keep), dtype=np.int32)
    for b in range(B):
        forced = set(range(min(n_sink, T))) | set(range(max(0, T - n_recent), T))
        rest = sorted((t for t in range(T) if t not in forced), key=lambda t: (-M[b, t], t))
        chosen = sorted(forced | set(rest[:T_keep - len(forced)]))
        keep[b] = chosen
    return keep

"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each test checks the oracle against one of: a hand-worked example under tests/golden (with its
derivation), a library routine that computes the same closed form (torch scaled_dot_product_attention,
torch/numpy format conversions, numpy complex exponentials), an invariant of the mathematics (rotation
identities, the full-rank round trip), or brute force on tiny inputs.  Together they are chosen so that
a dropped term, a wrong sign, a wrong index or a transposed operand anywhere in the oracle fails one.

Method passages (web pages about arXiv:2611.07025, cited by title and section):
  "LowRAM: Low-Rank Keys and Amortised Values for Composable KV Cache Compression at Test-Time", Abstract
  "LowRAM Paper: Amortised Values and Low-Rank Keys for KV Compression": "Value cache amortisation in
  plain language", "Asymmetric key compression with xKV", "Step-by-step mental model for one decoding session"
  "LowRAM: predict values from keys, store only the misses": flowchart "Values are mostly a function of keys"
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle as O

RNG = np.random.default_rng(12345)


# ------------------------------------------------------------------------------------------------
# independent helpers (library routines, not the oracle's code)
# ------------------------------------------------------------------------------------------------
def rope_complex(x, pos, theta):
    """Rotary embedding as a complex multiplication: feature pair (i, i+d/2) is the complex number
    x_i + j x_{i+d/2}, multiplied by exp(j * pos * theta^(-2i/d))."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    z = x[..., :h] + 1j * x[..., h:]
    w = theta ** (-2.0 * np.arange(h) / d)
    z = z * np.exp(1j * np.asarray(pos, dtype=np.float64)[..., None] * w)
    return np.concatenate([z.real, z.imag], axis=-1)


def sdpa(q, k, v, mask=None, scale=None):
    """torch fp64 scaled_dot_product_attention for one query per q-head.
    q [B,Hq,d], k/v [B,T,Hkv,d]; mask [B,Hkv,T] bool (True = attend)."""
    Q = torch.as_tensor(q, dtype=torch.float64)[:, :, None, :]
    K = torch.as_tensor(k, dtype=torch.float64).permute(0, 2, 1, 3)
    V = torch.as_tensor(v, dtype=torch.float64).permute(0, 2, 1, 3)
    g = Q.shape[1] // K.shape[1]
    am = None
    if mask is not None:
        am = torch.as_tensor(mask).repeat_interleave(g, dim=1)[:, :, None, :]
    out = F.scaled_dot_product_attention(Q, K, V, attn_mask=am, scale=scale, enable_gqa=True)
    return out[:, :, 0, :].numpy()


def torch_logits(q, k_rot, scale):
    """[B,Hq,T] scaled logits via torch einsum with the kv-head of each q-head repeated."""
    Q = torch.as_tensor(q, dtype=torch.float64)
    K = torch.as_tensor(k_rot, dtype=torch.float64)
    g = Q.shape[1] // K.shape[2]
    K = K.repeat_interleave(g, dim=2)
    return (torch.einsum("bhd,bthd->bht", Q, K) * scale).numpy()


def full_rank_group(B=2, T=40, H_q=4, H_kv=2, d=8, G=2, m=6, seed=0):
    """A layer group whose stacked basis is square (r = G*H_kv*d) and invertible, with original keys and
    values drawn directly (not from any latent)."""
    rng = np.random.default_rng(seed)
    N = G * H_kv * d
    r = N
    W_stack = rng.normal(0, r ** -0.5, (N, r)) + np.eye(N) * 0.5
    bases = [W_stack[l * H_kv * d:(l + 1) * H_kv * d] for l in range(G)]
    proj = np.linalg.inv(W_stack)                       # proj @ W_stack = I
    k_cat = rng.normal(0, 1, (B, T, N))
    vs = [rng.normal(0, 1, (B, T, H_kv, d)) for _ in range(G)]
    w1s = [rng.normal(0, d ** -0.5, (H_kv, m, d)) for _ in range(G)]
    w2s = [rng.normal(0, m ** -0.5, (H_kv, d, m)) for _ in range(G)]
    q = rng.normal(0, d ** -0.5, (B, H_q, d))
    return dict(B=B, T=T, H_q=H_q, H_kv=H_kv, d=d, G=G, m=m, r=r, bases=bases, proj=proj, k_cat=k_cat, vs=vs,
                w1s=w1s, w2s=w2s, q=q)


# ------------------------------------------------------------------------------------------------
# storage formats
# ------------------------------------------------------------------------------------------------
def test_bf16_rounding_matches_torch_on_float32_values():
    x = RNG.normal(0, 3, 20000).astype(np.float32)
    x = np.concatenate([x, np.float32([1e-39, -3e-40, 1e38, 65504.0, 0.0, -0.0])])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.round_bf16(x.astype(np.float64)), want)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1.0); 1 + 3*2^-8 -> 1 + 2^-6 (even mantissa)
    x = np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -8 + 2 ** -30])
    np.testing.assert_array_equal(O.round_bf16(x), [1.0, 1 + 2 ** -6, -1.0, 1 + 2 ** -7])


def test_f16_rounding_matches_numpy():
    x = np.concatenate([RNG.normal(0, 1, 5000), RNG.normal(0, 1e-5, 500), [65504.0, 65519.0, 1e-8]])
    np.testing.assert_array_equal(O.round_f16(x), x.astype(np.float16).astype(np.float64))


def test_int4_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "int4_group.json")))
    x = np.array(g["x"])[None, :]
    packed, scales = O.quant_int4_g32(x)
    np.testing.assert_array_equal(scales[0], g["scales"])
    np.testing.assert_array_equal(packed[0, :16], g["packed_group0"])
    deq = O.dequant_int4_g32(packed, scales)[0]
    np.testing.assert_array_equal(deq, np.array(g["codes"]) * np.repeat(g["scales"], 32))


def test_int4_round_trip_bound_and_range():
    x = RNG.normal(0, 1, (64, 128))
    packed, scales = O.quant_int4_g32(x)
    deq = O.dequant_int4_g32(packed, scales)
    s = np.repeat(scales, 32, axis=1)
    assert np.all(np.abs(x - deq) <= s / 2 * (1 + 1e-3) + 1e-12)
    codes = np.where(s > 0, np.round(deq / np.where(s > 0, s, 1)), 0)
    assert codes.min() >= -7 and codes.max() <= 7
    # the largest entry of each group is within half a step of +-7 steps (scale is amax/7 rounded to fp16)
    amax = np.abs(x).reshape(64, 4, 32).max(-1)
    np.testing.assert_allclose(scales, np.float16(amax / 7).astype(np.float64))


def test_int8_golden_and_bound(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "int8_vec.json")))
    codes, sc = O.quant_int8_vec(np.array(g["x"])[None])
    assert sc[0] == g["scale"]
    np.testing.assert_array_equal(codes[0], g["codes"])
    x = RNG.normal(0, 0.3, (100, 64))
    codes, sc = O.quant_int8_vec(x)
    deq = O.dequant_int8_vec(codes, sc)
    assert np.all(np.abs(x - deq) <= sc[:, None] / 2 * (1 + 1e-3) + 1e-12)
    assert np.abs(codes.astype(int)).max() <= 127


# ------------------------------------------------------------------------------------------------
# RoPE
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("d,theta", [(2, 1e4), (8, 1e4), (64, 5e5), (128, 1e6)])
def test_rope_matches_complex_rotation(d, theta):
    x = RNG.normal(0, 1, d)
    for pos in [0, 1, 7, 1000, 65535]:
        np.testing.assert_allclose(O.rope(x, pos, theta), rope_complex(x, pos, theta), rtol=0, atol=1e-10)


def test_rope_angles_closed_form():
    c, s = O.rope_angles(4, 100.0, 3.0)           # w = [1, 100^-0.5 = 0.1]
    np.testing.assert_allclose(c, [math.cos(3.0), math.cos(0.3)], atol=1e-15)
    np.testing.assert_allclose(s, [math.sin(3.0), math.sin(0.3)], atol=1e-15)


def test_rope_relative_position_identity_norm_and_inverse():
    d, theta = 16, 1e4
    q, k = RNG.normal(0, 1, d), RNG.normal(0, 1, d)
    for a, b in [(0, 5), (17, 3), (1000, 1234)]:
        lhs = O.rope(q, a, theta) @ O.rope(k, b, theta)
        rhs = q @ O.rope(k, b - a, theta)
        assert abs(lhs - rhs) < 1e-10
        assert abs(np.linalg.norm(O.rope(k, b, theta)) - np.linalg.norm(k)) < 1e-12
        np.testing.assert_allclose(O.rope(O.rope(k, b, theta), b, theta, inverse=True), k, atol=1e-12)


# ------------------------------------------------------------------------------------------------
# predictor
# ------------------------------------------------------------------------------------------------
def test_mlp_golden(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "mlp_tiny.json")))
    v = O.mlp(g["k"], g["w1"], g["b1"], g["w2"], g["b2"])
    np.testing.assert_allclose(v, g["v"], rtol=0, atol=1e-15)
    # no biases: v = w2 silu(w1 k)
    v0 = O.mlp(g["k"], g["w1"], None, g["w2"], None)
    h = np.array([1.0, -2.0, -1.0])
    h = h / (1 + np.exp(-h))
    np.testing.assert_allclose(v0, np.array(g["w2"]) @ h, atol=1e-15)


def test_predict_values_matches_single_mlp_per_head():
    B, T, H, d, m = 2, 5, 3, 4, 6
    k = RNG.normal(0, 1, (B, T, H, d))
    w1, w2 = RNG.normal(0, 1, (H, m, d)), RNG.normal(0, 1, (H, d, m))
    b1, b2 = RNG.normal(0, 1, (H, m)), RNG.normal(0, 1, (H, d))
    v = O.predict_values(k, w1, w2, b1, b2)
    for (b, t, h) in [(0, 0, 0), (1, 4, 2), (0, 3, 1)]:
        np.testing.assert_allclose(v[b, t, h], O.mlp(k[b, t, h], w1[h], b1[h], w2[h], b2[h]), atol=1e-14)
    # against torch's silu/linear on one head
    kt = torch.as_tensor(k[1, 2, 1])
    ref = F.linear(F.silu(F.linear(kt, torch.as_tensor(w1[1]), torch.as_tensor(b1[1]))), torch.as_tensor(w2[1]),
                   torch.as_tensor(b2[1])).numpy()
    np.testing.assert_allclose(v[1, 2, 1], ref, atol=1e-13)


# ------------------------------------------------------------------------------------------------
# key rebuild and projection
# ------------------------------------------------------------------------------------------------
def test_rebuild_keys_matches_matmul():
    B, T, H, d, r = 2, 7, 3, 4, 10
    C, W = RNG.normal(0, 1, (B, T, r)), RNG.normal(0, 1, (H * d, r))
    k = O.rebuild_keys(C, W, H, d)
    np.testing.assert_allclose(k.reshape(B, T, H * d), np.matmul(C, W.T), atol=1e-12)


def test_project_recovers_latents_with_pinv():
    # keys exactly low rank: K = C0 . W_stack^T with N > r; proj = pinv(W_stack) -> C0 back
    B, T, G, H, d, r = 2, 9, 3, 2, 4, 7
    N = G * H * d
    W_stack = RNG.normal(0, 1, (N, r))
    C0 = RNG.normal(0, 1, (B, T, r))
    K = np.matmul(C0, W_stack.T)
    C = O.project(K, np.linalg.pinv(W_stack), G, H, d)
    np.testing.assert_allclose(C, C0, atol=1e-10)
    # keys handed over after RoPE at scattered positions: the oracle rotates them back first
    pos = np.stack([np.sort(RNG.choice(5000, T, replace=False)) for _ in range(B)]).astype(np.int32)
    K_rot = rope_complex(K.reshape(B, T, G * H, d), pos[:, :, None], 1e4).reshape(B, T, N)
    C2 = O.project(K_rot, np.linalg.pinv(W_stack), G, H, d, pos=pos, keys_post_rope=True, theta=1e4)
    np.testing.assert_allclose(C2, C0, atol=1e-9)


# ------------------------------------------------------------------------------------------------
# the whole path: full rank, every residual kept, S = T  ==  textbook attention on the original K, V
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("use_pos", [False, True])
def test_full_rank_all_residuals_no_selection_equals_sdpa(use_pos):
    g = full_rank_group()
    B, T, H_q, H_kv, d, G = g["B"], g["T"], g["H_q"], g["H_kv"], g["d"], g["G"]
    theta = 1e4
    pos = None
    if use_pos:  # evicted cache: kept tokens at scattered original positions
        pos = np.stack([np.sort(RNG.choice(3 * T, T, replace=False)) for _ in range(B)]).astype(np.int32)
    comp = O.compress_group(g["k_cat"], g["vs"], g["proj"], g["bases"], g["w1s"], g["w2s"], G=G, H_kv=H_kv, d=d,
                            n_res=T, coef_fmt="f64", res_fmt="f64")
    for l in range(G):
        k_orig = g["k_cat"].reshape(B, T, G, H_kv, d)[:, :, l]
        p = np.arange(T)[None, :].repeat(B, 0) if pos is None else pos
        k_rot = rope_complex(k_orig, p[:, :, None], theta)
        want = sdpa(g["q"], k_rot, g["vs"][l])
        lay = comp["layers"][l]
        res = O.decode(g["q"], comp["coef"], g["bases"][l], g["w1s"][l], g["w2s"][l], S=T, theta=theta, pos=pos,
                       res_idx=lay["res_idx"], res_val=lay["res_val"])
        np.testing.assert_allclose(res.out, want, rtol=0, atol=1e-10)
        logits = torch_logits(g["q"], k_rot, d ** -0.5)
        np.testing.assert_allclose(res.lse, torch.logsumexp(torch.as_tensor(logits), -1).numpy(), atol=1e-10)


def test_no_residuals_is_pure_predictor_attention():
    g = full_rank_group(seed=3)
    B, T, H_q, H_kv, d, G = g["B"], g["T"], g["H_q"], g["H_kv"], g["d"], g["G"]
    C = O.project(g["k_cat"], g["proj"], G, H_kv, d)
    k_pre = O.rebuild_keys(C, g["bases"][0], H_kv, d)
    np.testing.assert_allclose(k_pre, g["k_cat"].reshape(B, T, G, H_kv, d)[:, :, 0], atol=1e-10)
    vhat = O.predict_values(k_pre, g["w1s"][0], g["w2s"][0])
    k_rot = rope_complex(k_pre, np.arange(T)[None, :, None], 1e4)
    res = O.decode(g["q"], C, g["bases"][0], g["w1s"][0], g["w2s"][0], S=T, theta=1e4)
    np.testing.assert_allclose(res.out, sdpa(g["q"], k_rot, vhat), atol=1e-11)


# ------------------------------------------------------------------------------------------------
# selection
# ------------------------------------------------------------------------------------------------
def _decode_case(S, seed=5, T=37, n_res=9, pos=None):
    rng = np.random.default_rng(seed)
    B, H_q, H_kv, d, r, m = 2, 6, 2, 8, 5, 7
    C = rng.normal(0, 1, (B, T, r))
    W = rng.normal(0, r ** -0.5, (H_kv * d, r))
    w1, w2 = rng.normal(0, d ** -0.5, (H_kv, m, d)), rng.normal(0, m ** -0.5, (H_kv, d, m))
    b1, b2 = rng.normal(0, 0.1, (H_kv, m)), rng.normal(0, 0.1, (H_kv, d))
    q = rng.normal(0, 1, (B, H_q, d))
    ridx = np.stack([[np.sort(rng.choice(T, n_res, replace=False)) for _ in range(H_kv)] for _ in range(B)])
    rval = rng.normal(0, 0.3, (B, H_kv, n_res, d))
    res = O.decode(q, C, W, w1, w2, b1=b1, b2=b2, S=S, theta=1e4, pos=pos, res_idx=ridx, res_val=rval)
    return dict(B=B, T=T, H_q=H_q, H_kv=H_kv, d=d, C=C, W=W, w1=w1, w2=w2, b1=b1, b2=b2, q=q, ridx=ridx,
                rval=rval, res=res, pos=pos)


def _explicit(c):
    """Explicit rotated keys and effective values (predictor + scattered residuals) of a decode case."""
    B, T, H_kv, d = c["B"], c["T"], c["H_kv"], c["d"]
    k_pre = np.matmul(c["C"], c["W"].T).reshape(B, T, H_kv, d)
    p = np.arange(T)[None, :].repeat(B, 0) if c["pos"] is None else c["pos"]
    k_rot = rope_complex(k_pre, p[:, :, None], 1e4)
    vhat = O.predict_values(k_pre, c["w1"], c["w2"], c["b1"], c["b2"])
    r_full = np.zeros_like(vhat)
    for b in range(B):
        for h in range(H_kv):
            r_full[b, c["ridx"][b, h], h] += c["rval"][b, h]
    return k_rot, vhat + r_full


@pytest.mark.parametrize("S", [1, 4, 16, 36, 37, 100])
def test_selection_brute_force_and_masked_attention(S):
    c = _decode_case(S)
    B, T, H_q, H_kv = c["B"], c["T"], c["H_q"], c["H_kv"]
    k_rot, v_eff = _explicit(c)
    logits = torch_logits(c["q"], k_rot, c["d"] ** -0.5)                 # [B, Hq, T]
    key = logits.reshape(B, H_kv, H_q // H_kv, T).max(2)
    np.testing.assert_allclose(c["res"].key, key, atol=1e-12)
    S_eff = min(S, T)
    mask = np.zeros((B, H_kv, T), dtype=bool)
    for b in range(B):
        for h in range(H_kv):
            order = sorted(range(T), key=lambda t: (-c["res"].key[b, h, t], t))[:S_eff]
            assert list(c["res"].sel[b, h]) == sorted(order)
            mask[b, h, order] = True
    np.testing.assert_allclose(c["res"].out, sdpa(c["q"], k_rot, v_eff, mask=mask), atol=1e-12)


def test_selection_of_one_returns_argmax_value():
    c = _decode_case(1)
    k_rot, v_eff = _explicit(c)
    for b in range(c["B"]):
        for h in range(c["H_kv"]):
            t = int(np.argmax(c["res"].key[b, h]))
            for jq in range(c["H_q"] // c["H_kv"]):
                np.testing.assert_allclose(c["res"].out[b, h * (c["H_q"] // c["H_kv"]) + jq], v_eff[b, t, h],
                                           atol=1e-13)


def test_selection_ties_go_to_lower_index():
    # two tokens get identical latents and the same position, so identical keys in every head
    rng = np.random.default_rng(9)
    T = 30
    pos = np.arange(T, dtype=np.int32)[None, :].copy()
    tie_a, tie_b = 3, 4
    pos[0, tie_b] = pos[0, tie_a]       # tokens 3 and 4 share position 3 (positions stay ascending)
    C = rng.normal(0, 1, (1, T, 4))
    C[0, tie_b] = C[0, tie_a]
    W = rng.normal(0, 0.5, (1 * 4, 4))
    w1, w2 = rng.normal(0, 0.5, (1, 3, 4)), rng.normal(0, 0.5, (1, 4, 3))
    q = rng.normal(0, 1, (1, 2, 4))
    full = O.decode(q, C, W, w1, w2, S=T, theta=1e4, pos=pos)
    key = full.key[0, 0]
    assert key[tie_a] == key[tie_b]
    rank = sorted(range(T), key=lambda t: (-key[t], t)).index(tie_a)
    sel = O.decode(q, C, W, w1, w2, S=rank + 1, theta=1e4, pos=pos).sel[0, 0]
    assert tie_a in sel and tie_b not in sel


def test_eviction_positions_are_used():
    pos = np.stack([np.sort(np.random.default_rng(1).choice(500, 37, replace=False))] * 2).astype(np.int32)
    c = _decode_case(12, pos=pos)
    k_rot, v_eff = _explicit(c)
    logits = torch_logits(c["q"], k_rot, c["d"] ** -0.5)
    np.testing.assert_allclose(c["res"].key, logits.reshape(2, 2, 3, 37).max(2), atol=1e-12)


# ------------------------------------------------------------------------------------------------
# write side: worst-token residuals
# ------------------------------------------------------------------------------------------------
def _planted(T=50, n_res=7, seed=2, ties=False):
    rng = np.random.default_rng(seed)
    B, H, d, r, m = 2, 2, 6, 4, 5
    C = rng.normal(0, 1, (B, T, r))
    W = rng.normal(0, 0.5, (H * d, r))
    w1, w2 = rng.normal(0, 0.5, (H, m, d)), rng.normal(0, 0.5, (H, d, m))
    vhat = O.predict_values(np.matmul(C, W.T).reshape(B, T, H, d), w1, w2)
    e = rng.permutation(np.linspace(0.1, 5.0, B * T * H)).reshape(B, H, T)   # distinct planted errors
    if ties:
        e[0, 0, 11] = e[0, 0, 30] = 100.0
    u = rng.normal(0, 1, (B, T, H, d))
    u /= np.linalg.norm(u, axis=-1, keepdims=True)
    delta = u * e.transpose(0, 2, 1)[..., None]
    return C, W, w1, w2, vhat + delta, delta, e


def test_residuals_keep_the_planted_worst_tokens():
    C, W, w1, w2, V, delta, e = _planted()
    ridx, rraw, err = O.residuals(C, V, W, w1, w2, 7)
    np.testing.assert_allclose(err, e, atol=1e-12)
    for b in range(2):
        for h in range(2):
            want = sorted(sorted(range(50), key=lambda t: (-e[b, h, t], t))[:7])
            assert list(ridx[b, h]) == want
            np.testing.assert_allclose(rraw[b, h], delta[b, want, h], atol=1e-12)


def test_residual_ties_go_to_lower_index():
    C, W, w1, w2, V, delta, e = _planted(ties=True)
    ridx, _, _ = O.residuals(C, V, W, w1, w2, 1)
    assert ridx[0, 0, 0] == 11


def test_all_residuals_reconstruct_values_exactly():
    C, W, w1, w2, V, delta, e = _planted()
    ridx, rraw, _ = O.residuals(C, V, W, w1, w2, 50)
    vhat = O.predict_values(np.matmul(C, W.T).reshape(2, 50, 2, 6), w1, w2)
    for b in range(2):
        for h in range(2):
            assert list(ridx[b, h]) == list(range(50))
            np.testing.assert_allclose(vhat[b, :, h] + rraw[b, h], V[b, :, h], atol=1e-12)
    ridx0, rraw0, _ = O.residuals(C, V, W, w1, w2, 0)
    assert ridx0.shape == (2, 2, 0)


# ------------------------------------------------------------------------------------------------
# comparator and budgets
# ------------------------------------------------------------------------------------------------
def test_dense_decode_matches_sdpa():
    B, T, H_q, H_kv, d = 2, 33, 8, 2, 16
    q, k, v = RNG.normal(0, 1, (B, H_q, d)), RNG.normal(0, 1, (B, T, H_kv, d)), RNG.normal(0, 1, (B, T, H_kv, d))
    out, lse = O.dense_decode(q, k, v)
    np.testing.assert_allclose(out, sdpa(q, k, v), atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.as_tensor(torch_logits(q, k, d ** -0.5)), -1).numpy(),
                               atol=1e-12)


# ------------------------------------------------------------------------------------------------
# exact tail: body and tail attended separately, merged through their log-sum-exp
# ------------------------------------------------------------------------------------------------
@pytest.mark.parametrize("cut", [1, 17, 32])
def test_merge_of_a_split_equals_attention_over_the_union(cut):
    B, T, H_q, H_kv, d = 2, 33, 8, 2, 16
    q, k, v = RNG.normal(0, 1, (B, H_q, d)), RNG.normal(0, 2, (B, T, H_kv, d)), RNG.normal(0, 1, (B, T, H_kv, d))
    oa, la = O.dense_decode(q, k[:, :cut], v[:, :cut])
    ob, lb = O.dense_decode(q, k[:, cut:], v[:, cut:])
    out, lse = O.merge_attn(oa, la, ob, lb)
    np.testing.assert_allclose(out, sdpa(q, k, v), atol=1e-12)
    np.testing.assert_allclose(lse, torch.logsumexp(torch.as_tensor(torch_logits(q, k, d ** -0.5)), -1).numpy(),
                               atol=1e-12)
    out2, lse2 = O.merge_attn(ob, lb, oa, la)          # order of the two sets does not matter
    np.testing.assert_allclose(out2, out, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, atol=1e-14)


def test_merge_with_empty_sets():
    o = RNG.normal(0, 1, (2, 3, 4))
    l = RNG.normal(0, 1, (2, 3))
    ninf = np.full((2, 3), -np.inf)
    out, lse = O.merge_attn(o, l, np.zeros_like(o), ninf)
    np.testing.assert_array_equal(out, o)
    np.testing.assert_array_equal(lse, l)
    out, lse = O.merge_attn(np.zeros_like(o), ninf, np.zeros_like(o), ninf)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_compressed_body_plus_exact_tail_equals_sdpa_over_everything():
    """Full rank, every residual kept, S = T: the body is exact, so body + tail merged is textbook attention over
    the prompt's tokens followed by the explicitly kept decoded tokens."""
    g = full_rank_group(seed=7)
    B, T, H_q, H_kv, d, G = g["B"], g["T"], g["H_q"], g["H_kv"], g["d"], g["G"]
    theta, n_tail = 1e4, 5
    comp = O.compress_group(g["k_cat"], g["vs"], g["proj"], g["bases"], g["w1s"], g["w2s"], G=G, H_kv=H_kv, d=d,
                            n_res=T, coef_fmt="f64", res_fmt="f64")
    l = 1
    k_body = rope_complex(g["k_cat"].reshape(B, T, G, H_kv, d)[:, :, l], np.arange(T)[None, :, None], theta)
    k_tail_pre = RNG.normal(0, 1, (B, n_tail, H_kv, d))
    k_tail = rope_complex(k_tail_pre, np.arange(T, T + n_tail)[None, :, None], theta)
    v_tail = RNG.normal(0, 1, (B, n_tail, H_kv, d))
    lay = comp["layers"][l]
    body = O.decode(g["q"], comp["coef"], g["bases"][l], g["w1s"][l], g["w2s"][l], S=T, theta=theta,
                    res_idx=lay["res_idx"], res_val=lay["res_val"])
    ot, lt = O.dense_decode(g["q"], k_tail, v_tail)
    out, lse = O.merge_attn(body.out, body.lse, ot, lt)
    k_all = np.concatenate([k_body, k_tail], axis=1)
    v_all = np.concatenate([g["vs"][l], v_tail], axis=1)
    np.testing.assert_allclose(out, sdpa(g["q"], k_all, v_all), rtol=0, atol=1e-10)


# ------------------------------------------------------------------------------------------------
# fitted basis (cross-layer SVD of the RoPE-inverted keys)
# ------------------------------------------------------------------------------------------------
def low_rank_keys(B, T, D, r, noise, seed):
    rng = np.random.default_rng(seed)
    U, _ = np.linalg.qr(rng.normal(0, 1, (D, r)))
    sig = np.geomspace(10.0, 1.0, r)                     # decaying spectrum, well above the noise
    C = rng.normal(0, 1, (B * T, r)) * sig
    return (C @ U.T + noise * rng.normal(0, 1, (B * T, D))).reshape(B, T, D)


def test_fit_basis_is_exact_for_low_rank_keys():
    B, T, G, H_kv, d, r = 2, 50, 2, 2, 8, 6
    K = low_rank_keys(B, T, G * H_kv * d, r, 0.0, 1)
    proj, bases, w = O.fit_basis(K, r, G, H_kv, d)
    Wst = np.concatenate(bases, axis=0)
    np.testing.assert_allclose(proj @ Wst, np.eye(r), atol=1e-12)             # proj is a left inverse
    Kf = K.reshape(B * T, -1)
    np.testing.assert_allclose(Kf @ proj.T @ Wst.T, Kf, atol=1e-9)              # rank r keys are rebuilt
    assert np.all(np.diff(w) <= 0)


def test_fit_basis_meets_eckart_young():
    """Rebuild error of the fitted subspace = the norm of the discarded singular values (numpy SVD of the keys
    themselves, not of the Gram matrix), and the subspace is the top-r right singular subspace."""
    B, T, G, H_kv, d, r = 2, 60, 2, 2, 8, 5
    K = low_rank_keys(B, T, G * H_kv * d, r, 0.3, 2)
    proj, bases, _ = O.fit_basis(K, r, G, H_kv, d)
    Kf = K.reshape(B * T, -1)
    s = np.linalg.svd(Kf, compute_uv=False)
    err = np.linalg.norm(Kf - Kf @ proj.T @ proj)
    assert abs(err - math.sqrt(float(np.sum(s[r:] ** 2)))) <= 1e-9 * err
    Vt = np.linalg.svd(Kf, full_matrices=False)[2][:r]
    np.testing.assert_allclose(proj.T @ proj, Vt.T @ Vt, atol=1e-9)


def test_fit_basis_inverts_rope_of_rotated_keys():
    B, T, G, H_kv, d, r, theta = 2, 40, 2, 2, 8, 5, 1e4
    K = low_rank_keys(B, T, G * H_kv * d, r, 0.1, 3).reshape(B, T, G, H_kv, d)
    pos = np.stack([np.sort(RNG.choice(200, T, replace=False)) for _ in range(B)]).astype(np.int32)
    K_rot = rope_complex(K, pos[:, :, None, None], theta)
    p1, _, w1 = O.fit_basis(K, r, G, H_kv, d)
    p2, _, w2 = O.fit_basis(K_rot, r, G, H_kv, d, pos=pos, keys_post_rope=True, theta=theta)
    np.testing.assert_allclose(w2, w1, rtol=1e-10)
    np.testing.assert_allclose(p2.T @ p2, p1.T @ p1, atol=1e-9)


# ------------------------------------------------------------------------------------------------
# test-time fit of the predictor: loss gradient and Adam
# ------------------------------------------------------------------------------------------------
def predictor_params(d, m, seed):
    rng = np.random.default_rng(seed)
    return (rng.normal(0, d ** -0.5, (m, d)), rng.normal(0, 0.1, m), rng.normal(0, m ** -0.5, (d, m)),
            rng.normal(0, 0.1, d))


def test_predictor_loss_is_the_mse_of_the_oracle_mlp():
    N, d, m = 7, 4, 6
    rng = np.random.default_rng(8)
    K, V = rng.normal(0, 1, (N, d)), rng.normal(0, 1, (N, d))
    w1, b1, w2, b2 = predictor_params(d, m, 9)
    loss = O.predictor_loss_grad(K, V, w1, b1, w2, b2)[0]
    want = np.mean([(O.mlp(K[t], w1, b1, w2, b2) - V[t]) ** 2 for t in range(N)])
    assert abs(loss - want) <= 1e-14


def test_predictor_gradient_matches_central_differences():
    N, d, m = 9, 5, 4
    rng = np.random.default_rng(10)
    K, V = rng.normal(0, 1, (N, d)), rng.normal(0, 1, (N, d))
    params = list(predictor_params(d, m, 11))
    _, *grads = O.predictor_loss_grad(K, V, *params)
    h = 1e-6
    for i, (p, g) in enumerate(zip(params, grads)):
        num = np.zeros_like(p)
        for idx in np.ndindex(p.shape):
            plus = [x.copy() for x in params]
            minus = [x.copy() for x in params]
            plus[i][idx] += h
            minus[i][idx] -= h
            num[idx] = (O.predictor_loss_grad(K, V, *plus)[0] - O.predictor_loss_grad(K, V, *minus)[0]) / (2 * h)
        np.testing.assert_allclose(g, num, atol=1e-8, rtol=1e-6)


def test_adam_first_steps_closed_form():
    """Adam's first step moves each parameter by lr * sign(g) (up to eps); a constant gradient keeps that step."""
    p, g = np.array([1.0, -2.0, 0.5]), np.array([0.3, -4.0, 1e-3])
    p1, m, v = O.adam_step(p, g, 0.0, 0.0, 1, 0.01, 0.9, 0.999, 1e-12)
    np.testing.assert_allclose(p1, p - 0.01 * np.sign(g), atol=1e-10)
    p2, _, _ = O.adam_step(p1, g, m, v, 2, 0.01, 0.9, 0.999, 1e-12)
    np.testing.assert_allclose(p2, p1 - 0.01 * np.sign(g), atol=1e-10)


def test_fit_predictor_recovers_a_planted_predictor():
    """Values generated by a predictor of the same shape: the fit's loss falls by orders of magnitude."""
    B, T, H_kv, d, m = 1, 200, 2, 4, 8
    rng = np.random.default_rng(12)
    K = rng.normal(0, 1, (B, T, H_kv, d))
    true = [predictor_params(d, m, 20 + h) for h in range(H_kv)]
    V = np.stack([np.stack([O.mlp(K[0, t, h], *true[h]) for t in range(T)]) for h in range(H_kv)], axis=1)[None]
    start = [np.stack(x) for x in zip(*[predictor_params(d, m, 40 + h) for h in range(H_kv)])]
    *_, losses = O.fit_predictor(K, V, *start, steps=400, lr=0.02)
    assert np.all(losses[-1] < 1e-2 * losses[0])
    assert np.all(np.diff(losses[:50], axis=0) < 0)     # early steps descend


# ------------------------------------------------------------------------------------------------
# heavy hitters from accumulated attention (eviction)
# ------------------------------------------------------------------------------------------------
def test_attention_mass_matches_torch_softmax_and_sums_to_the_window():
    B, W, H_q, H_kv, T, d = 2, 3, 4, 2, 17, 8
    q, k = RNG.normal(0, 1, (B, W, H_q, d)), RNG.normal(0, 1, (B, T, H_kv, d))
    mass = O.attention_mass(q, k)
    want = np.zeros((B, T))
    for b in range(B):
        for hq in range(H_q):
            lg = torch.as_tensor(q[b, :, hq]) @ torch.as_tensor(k[b, :, hq // 2]).T * d ** -0.5
            want[b] += torch.softmax(lg, dim=-1).sum(0).numpy()
    np.testing.assert_allclose(mass, want, atol=1e-12)
    np.testing.assert_allclose(mass.sum(axis=1), W * H_q, atol=1e-10)


def test_attention_mass_closed_form_and_head_grouping():
    """kv-head 0 holds one key repeated, so its q-heads attend uniformly (1/T per token); kv-head 1 holds zero keys
    except a large multiple of the shared direction u of its q-heads at token 5, so each of those rows puts
    p5 = e^s / (e^s + T - 1) on token 5 and (1 - p5)/(T - 1) elsewhere.  A q-head to kv-head map other than
    hq // g breaks the sum."""
    W, H_q, H_kv, T, d = 2, 4, 2, 9, 8
    g = H_q // H_kv
    u = RNG.normal(0, 1, d)
    q = RNG.normal(0, 1, (1, W, H_q, d))
    q[0, :, 2:] = u                                           # kv-head 1's q-heads
    k = np.zeros((1, T, H_kv, d))
    k[0, :, 0] = RNG.normal(0, 1, d)
    k[0, 5, 1] = 0.5 * u
    s = 0.5 * (u @ u) * d ** -0.5
    p5 = np.exp(s) / (np.exp(s) + T - 1)
    want = np.full(T, W * g / T + W * g * (1 - p5) / (T - 1))
    want[5] = W * g / T + W * g * p5
    np.testing.assert_allclose(O.attention_mass(q, k)[0], want, rtol=1e-12)


def test_evict_plan_keeps_sinks_recents_and_the_heaviest():
    T, n_sink, n_recent, T_keep = 30, 3, 5, 14
    mass = RNG.random((2, T))
    mass[1, 10] = mass[1, 11] = 5.0                   # a tie among the heaviest: both kept
    keep = O.evict_plan(mass, n_sink, n_recent, T_keep)
    for b in range(2):
        kb = keep[b].tolist()
        assert kb == sorted(kb) and len(set(kb)) == T_keep
        assert set(range(n_sink)) <= set(kb) and set(range(T - n_recent, T)) <= set(kb)
        middle = [t for t in range(n_sink, T - n_recent)]
        heavy = sorted(middle, key=lambda t: (-mass[b, t], t))[:T_keep - n_sink - n_recent]   # brute force
        assert set(kb) == set(range(n_sink)) | set(range(T - n_recent, T)) | set(heavy)
    assert {10, 11} <= set(keep[1].tolist())
    flat = np.ones((1, T))                               # all equal: the lowest middle indices win
    assert O.evict_plan(flat, n_sink, n_recent, T_keep)[0].tolist() == \
        list(range(n_sink + T_keep - n_sink - n_recent)) + list(range(T - n_recent, T))
    assert O.evict_plan(mass, n_sink, n_recent, T)[0].tolist() == list(range(T))


def test_residual_budgets_of_the_workloads():
    # ceil(rho * T): 0.25*256, 0.1*8192, 0.1*32768, 0.1*4096, 0.05*16384
    assert [O.n_res_for(r, T) for r, T in [(0.25, 256), (0.1, 8192), (0.1, 32768), (0.1, 4096), (0.05, 16384)]] \
        == [64, 820, 3277, 410, 820]
    assert O.n_res_for(0.0, 100) == 0 and O.n_res_for(1.0, 100) == 100


def test_empty_and_degenerate_shapes():
    rng = np.random.default_rng(0)
    q = rng.normal(0, 1, (1, 2, 4))
    W = rng.normal(0, 1, (4, 3))
    w1, w2 = rng.normal(0, 1, (1, 2, 4)), rng.normal(0, 1, (1, 4, 2))
    # T = 0: empty attention, lse = -inf, out = 0
    res = O.decode(q, np.zeros((1, 0, 3)), W, w1, w2, S=4, theta=1e4)
    assert res.sel.shape == (1, 1, 0) and np.all(res.out == 0) and np.all(np.isneginf(res.lse))
    # S = 0: nothing selected
    res = O.decode(q, rng.normal(0, 1, (1, 5, 3)), W, w1, w2, S=0, theta=1e4)
    assert res.sel.shape == (1, 1, 0) and np.all(res.out == 0)
    # B = 0
    res = O.decode(np.zeros((0, 2, 4)), np.zeros((0, 5, 3)), W, w1, w2, S=4, theta=1e4)
    assert res.out.shape == (0, 2, 4)


def test_selection_projection_copies_key_features_exactly():
    """A 0/1 selection projection makes the oracle's latent coefficients exact copies of the selected key
    features (no rounding anywhere), and its bases rebuild exactly those features with zeros elsewhere."""
    import lowram_cases as C
    from decode_attention_19_b300 import synth
    w = synth.WORKLOADS["llama8b"].with_(B=1, T=48, G=2, H_kv=2, r=64, S=48)
    c = C.exact_projection_case(w)
    orc = C.run_oracle_compress(c)
    sel = c["proj"].argmax(dim=1).numpy()
    keys = O.f64(c["keys"]).reshape(w.B, w.T, -1)
    assert np.array_equal(orc["coef_raw"], keys[:, :, sel])
    assert np.array_equal(orc["coef"], keys[:, :, sel])
    rows = w.H_kv * w.d
    for l in range(w.G):
        rebuilt = O.rebuild_keys(orc["coef"], c["bases"][l], w.H_kv, w.d).reshape(w.B, w.T, -1)
        want = np.zeros_like(rebuilt)
        mine = (sel >= l * rows) & (sel < (l + 1) * rows)
        want[:, :, sel[mine] - l * rows] = keys[:, :, sel[mine]]
        assert np.array_equal(rebuilt, want)


def test_per_sequence_bases_and_predictors_pair_with_their_sequence():
    """A basis and a predictor given per sequence are used with that sequence only: permuting sequence b's latent
    dimensions (in its coefficients and its basis together) and its hidden units (w1 rows, b1, w2 columns
    together) leaves every output as with the shared weights, while giving sequence 0 sequence 1's basis changes
    sequence 0's output and no other."""
    from decode_attention_19_b300 import synth
    w = synth.WORKLOADS["tiny"].with_(B=3, T=40, S=17, r=32, m=64)
    raw = synth.draw_group(w, 0, with_noise=False)
    q = synth.draw_query(w, 0)
    coef = O.f64(raw["coef"])
    W, W1, W2 = O.f64(raw["basis"][0]), O.f64(raw["w1"][0]), O.f64(raw["w2"][0])
    b1 = RNG.normal(0, 0.1, (w.H_kv, w.m))
    b2 = RNG.normal(0, 0.1, (w.H_kv, w.d))
    ref = O.decode(q, coef, W, W1, W2, S=w.S, theta=w.theta, b1=b1, b2=b2)
    perms_r = [RNG.permutation(w.r) for _ in range(w.B)]
    perms_m = [RNG.permutation(w.m) for _ in range(w.B)]
    coef_p = np.stack([coef[b][:, p] for b, p in enumerate(perms_r)])
    Wb = np.stack([W[:, p] for p in perms_r])
    W1b = np.stack([W1[:, p, :] for p in perms_m])
    b1b = np.stack([b1[:, p] for p in perms_m])
    W2b = np.stack([W2[:, :, p] for p in perms_m])
    b2b = np.stack([b2] * w.B)
    got = O.decode(q, coef_p, Wb, W1b, W2b, S=w.S, theta=w.theta, b1=b1b, b2=b2b)
    np.testing.assert_allclose(got.out, ref.out, atol=1e-12)
    np.testing.assert_allclose(got.key, ref.key, atol=1e-12)
    assert np.array_equal(got.sel, ref.sel)
    Wswap = np.stack([W * 1.5, W, W])
    sw = O.decode(q, coef, Wswap, W1, W2, S=w.S, theta=w.theta, b1=b1, b2=b2)
    assert not np.allclose(sw.out[0], ref.out[0])
    np.testing.assert_allclose(sw.out[1:], ref.out[1:], atol=1e-12)

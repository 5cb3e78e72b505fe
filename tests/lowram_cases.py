"""Shared case construction and comparison for the GPU parity tests.

Inputs come from the seeded generator (``decode_attention_19_b300.synth``); derived inputs that need the
method's arithmetic (true keys and values for the write side, stored int4/int8 codes of raw draws) are
composed with the oracle, never with the CUDA path.  Comparisons follow the bar the library is held to:
float outputs within max-abs / relative-L2 tolerances, selection and residual index sets identical except
for tokens whose oracle score (or error) lies within 1e-3 of the oracle's cut-off.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from decode_attention_19_b300 import synth

KEY_TOL = 1e-4       # |gpu key - oracle key|, selection keys (scaled logits)
# int4 caches reach the tensor cores as an fp16 copy of code * scale (2^-12 relative rounding): the oracle's keys
# from fp16-rounded coefficients differ from its exact ones by up to 7.9e-5 at these shapes, so int4 keys get twice
# the bf16 tolerance (the exact two-term split, LOWRAM_FLAG_INT4_EXACT_SPLIT, keeps KEY_TOL)
KEY_TOL_INT4_F16 = 2e-4
BAND = 1e-3          # index sets may differ only within this distance of the cut-off
OUT_MAX_ABS = 1e-2   # bf16 inputs, fp32 accumulation
OUT_REL_L2 = 5e-3

_TDT = {"f32": torch.float32, "bf16": torch.bfloat16}


def stored_coef(w: synth.Workload, coef_raw: torch.Tensor):
    """(stored tensor for the GPU, fp64 values for the oracle, scale tensor or None)."""
    if w.coef_fmt == "int4":
        packed, scales = O.quant_int4_g32(coef_raw)
        vals = O.dequant_int4_g32(packed, scales)
        return torch.from_numpy(packed), vals, torch.from_numpy(scales).to(torch.float16)
    t = coef_raw.to(_TDT[w.coef_fmt])
    return t, O.f64(t), None


def stored_res(w: synth.Workload, res_raw):
    if w.res_fmt == "int8":
        codes, scales = O.quant_int8_vec(res_raw)
        return torch.from_numpy(codes), O.dequant_int8_vec(codes, scales), torch.from_numpy(scales).to(torch.float16)
    t = torch.as_tensor(np.asarray(O.f64(res_raw))).to(_TDT[w.res_fmt])
    return t, O.f64(t), None


def decode_case(w: synth.Workload, layer: int = 0, biases: bool = False) -> dict:
    raw = synth.draw_group(w, 0, with_noise=False)
    coef, coef_vals, coef_scale = stored_coef(w, raw["coef"])
    ridx, rval_raw = synth.placeholder_residuals(w, layer)
    res_val, res_vals64, res_scale = stored_res(w, rval_raw)
    c = dict(w=w, coef=coef, coef_vals=coef_vals, coef_scale=coef_scale, basis=raw["basis"][layer],
             w1=raw["w1"][layer], w2=raw["w2"][layer], q=synth.draw_query(w, layer), res_idx=ridx, res_val=res_val,
             res_vals64=res_vals64, res_scale=res_scale, pos=synth.eviction_positions(w) if w.T_nominal else None,
             b1=None, b2=None)
    if biases:
        c["b1"] = synth.gaussian((w.H_kv, w.m), 0.1, w.seed, w.name, "b1", layer)
        c["b2"] = synth.gaussian((w.H_kv, w.d), 0.1, w.seed, w.name, "b2", layer)
    c["max_pos"] = w.T_nominal if w.T_nominal else max(w.T, 1)
    return c


def run_gpu_decode(c: dict, *, S=None, hooks=True, workspace=None, int4_exact_split=False):
    import decode_attention_19_b300 as L
    w = c["w"]
    S = w.S if S is None else S
    dev = torch.device("cuda")
    cu = lambda t: None if t is None else t.to(dev).contiguous()
    cos, sin = L.lowram_rope_table(w.d, w.theta, c["max_pos"])
    T = c["coef"].shape[1]
    B = c["q"].shape[0]
    S_eff = min(S, T)
    key = torch.empty((B, w.H_kv, T), dtype=torch.float32, device=dev) if hooks else None
    sel = torch.empty((B, w.H_kv, S_eff), dtype=torch.int32, device=dev) if hooks else None
    n_res = c["res_idx"].shape[-1]
    own_ws = workspace is None
    if own_ws:   # 64 MiB, plus room for an int4 cache's exact bf16 split (rank 2r) and the repeated basis
        extra = 4 * w.r * (B * T + w.H_kv * w.d) + 4096 if w.coef_fmt == "int4" else 0
        workspace = torch.zeros((1 << 26) + extra, dtype=torch.uint8, device=dev)
    out, lse = L.lowram_decode_attn(cu(c["q"]), cu(c["coef"]), cu(c["basis"]), cu(c["w1"]), cu(c["w2"]),
                                    rope_cos=cos, rope_sin=sin, S=S, coef_scale=cu(c["coef_scale"]), pos=cu(c["pos"]),
                                    b1=cu(c["b1"]), b2=cu(c["b2"]),
                                    res_idx=cu(c["res_idx"]) if n_res else None,
                                    res_val=cu(c["res_val"]) if n_res else None,
                                    res_scale=cu(c["res_scale"]) if n_res else None, sel_out=sel, key_out=key,
                                    workspace=workspace, int4_exact_split=int4_exact_split)
    torch.cuda.synchronize()
    if own_ws:
        assert L.lowram_get_error(workspace) == 0, "device check word set"
    r = {"out": out.cpu().double().numpy(), "lse": lse.cpu().double().numpy(),
         "key_tol": KEY_TOL_INT4_F16 if (w.coef_fmt == "int4" and not int4_exact_split) else KEY_TOL}
    if hooks:
        r["key"] = key.cpu().double().numpy()
        r["sel"] = sel.cpu().numpy()
    return r


def slice_case(c: dict, bs, hs=None) -> dict:
    """Sub-problem of sequences bs and kv-heads hs (the oracle computes it independently of the rest)."""
    w = c["w"]
    g = w.H_q // w.H_kv
    hs = list(range(w.H_kv)) if hs is None else list(hs)
    qh = [h * g + j for h in hs for j in range(g)]
    rows = [h * w.d + i for h in hs for i in range(w.d)]
    s = dict(c)
    s["q"] = c["q"][bs][:, qh]
    s["coef_vals"] = c["coef_vals"][bs]
    s["basis"] = c["basis"][rows]
    s["w1"], s["w2"] = c["w1"][hs], c["w2"][hs]
    s["b1"] = None if c["b1"] is None else c["b1"][hs]
    s["b2"] = None if c["b2"] is None else c["b2"][hs]
    s["res_idx"] = c["res_idx"][bs][:, hs]
    s["res_vals64"] = c["res_vals64"][bs][:, hs]
    s["pos"] = None if c["pos"] is None else c["pos"][bs]
    return s


def run_oracle_decode(c: dict, *, S=None):
    w = c["w"]
    S = w.S if S is None else S
    n_res = c["res_idx"].shape[-1]
    return O.decode(c["q"], c["coef_vals"], c["basis"], c["w1"], c["w2"], S=S, theta=w.theta, pos=c["pos"],
                    b1=c["b1"], b2=c["b2"], res_idx=c["res_idx"] if n_res else None,
                    res_val=c["res_vals64"] if n_res else None)


def check_index_sets(gpu_sets, orc_sets, orc_vals, n_keep, band=BAND, allowed_extra=None, what="selection"):
    """gpu_sets/orc_sets [P, n] ascending indices; orc_vals [P, T] the oracle's ranking values."""
    P = orc_sets.shape[0]
    worst = 0
    for p in range(P):
        a, b = set(gpu_sets[p].tolist()), set(orc_sets[p].tolist())
        assert len(a) == len(gpu_sets[p]), f"{what}: duplicate indices in row {p}"
        assert list(gpu_sets[p]) == sorted(gpu_sets[p]), f"{what}: row {p} not ascending"
        diff = a ^ b
        if not diff:
            continue
        v = orc_vals[p]
        cut = np.sort(v)[::-1][n_keep - 1]
        for t in diff:
            if allowed_extra is not None and t in allowed_extra[p]:
                continue
            gap = abs(v[t] - cut)
            worst = max(worst, gap)
            assert gap <= band, f"{what}: row {p} token {t} differs, {gap:.3g} from the cut-off"
    return worst


def check_out(gpu_out, orc_out, max_abs=OUT_MAX_ABS, rel_l2=OUT_REL_L2):
    d = np.abs(gpu_out - orc_out)
    ma = float(d.max()) if d.size else 0.0
    nrm = float(np.linalg.norm(orc_out))
    rl = float(np.linalg.norm(gpu_out - orc_out) / nrm) if nrm > 0 else ma
    assert ma <= max_abs, f"max-abs {ma:.3g} > {max_abs}"
    assert rl <= rel_l2, f"rel-L2 {rl:.3g} > {rel_l2}"
    return ma, rl


def check_decode(gpu: dict, orc, S_eff: int, *, key_tol=None, max_abs=OUT_MAX_ABS, rel_l2=OUT_REL_L2):
    if key_tol is None:
        key_tol = gpu.get("key_tol", KEY_TOL)
    P = orc.key.shape[0] * orc.key.shape[1]
    if "key" in gpu:
        kd = np.abs(gpu["key"] - orc.key)
        assert float(kd.max()) <= key_tol, f"key max-abs {float(kd.max()):.3g}"
        if S_eff > 0:
            check_index_sets(gpu["sel"].reshape(P, -1), orc.sel.reshape(P, -1), orc.key.reshape(P, -1), S_eff)
    ma, rl = check_out(gpu["out"], orc.out, max_abs, rel_l2)
    if S_eff > 0:
        assert float(np.abs(gpu["lse"] - orc.lse).max()) <= 1e-3
    return ma, rl


# ------------------------------------------------------------------------------------------------
# write side
# ------------------------------------------------------------------------------------------------
def compress_case(w: synth.Workload, keys_post_rope: bool = False) -> dict:
    """True keys and values of one layer group, composed with the oracle from the generator's draws:
    keys_l = coef . basis_l (exactly low rank), values_l = predictor_l(keys_l) + N(0, 0.3^2) noise."""
    raw = synth.draw_group(w, 0, with_noise=True)
    act = _TDT[w.act]
    k_layers = [O.rebuild_keys(raw["coef"], raw["basis"][l], w.H_kv, w.d) for l in range(w.G)]
    v_layers = [O.predict_values(k_layers[l], raw["w1"][l], raw["w2"][l]) + O.f64(raw["noise"][l]) for l in range(w.G)]
    pos = synth.eviction_positions(w) if w.T_nominal else None
    keys64 = np.stack(k_layers, axis=2)                       # [B, T, G, H_kv, d]
    if keys_post_rope:
        P = np.arange(w.T)[None, :].repeat(w.B, 0) if pos is None else pos.numpy()
        keys64 = O.rope_rows(keys64, np.broadcast_to(P[:, :, None, None], keys64.shape[:-1]), w.theta)
    keys = torch.from_numpy(keys64).to(act)
    values = [torch.from_numpy(v).to(act) for v in v_layers]
    W_stack = np.concatenate([O.f64(b) for b in raw["basis"]], axis=0)        # [G*H_kv*d, r]
    proj = torch.from_numpy(np.linalg.pinv(W_stack)).to(torch.float32)     # proj . W_stack = I
    return dict(w=w, keys=keys, values=values, proj=proj, bases=raw["basis"], w1s=raw["w1"], w2s=raw["w2"], pos=pos,
                keys_post_rope=keys_post_rope, coef_raw_draw=raw["coef"])


def run_gpu_compress(c: dict) -> dict:
    import decode_attention_19_b300 as L
    w = c["w"]
    cu = lambda t: None if t is None else t.cuda().contiguous()
    fmt = {"f32": L.LOWRAM_F32, "bf16": L.LOWRAM_BF16, "int4": L.LOWRAM_INT4_G32, "int8": L.LOWRAM_INT8_VEC}
    cos = sin = None
    if c["keys_post_rope"]:
        cos, sin = L.lowram_rope_table(w.d, w.theta, w.T_nominal or max(w.T, 1))
    r = L.lowram_compress(cu(c["keys"]), [cu(v) for v in c["values"]], cu(c["proj"]), [cu(b) for b in c["bases"]],
                          [cu(x) for x in c["w1s"]], [cu(x) for x in c["w2s"]], n_res=w.n_res,
                          coef_dtype=fmt[w.coef_fmt], res_dtype=fmt[w.res_fmt], pos=cu(c["pos"]), rope_cos=cos,
                          rope_sin=sin, keys_post_rope=c["keys_post_rope"], want_err=True)
    torch.cuda.synchronize()
    return r


def run_oracle_compress(c: dict, bs=None) -> dict:
    w = c["w"]
    sl = slice(None) if bs is None else bs
    return O.compress_group(O.f64(c["keys"])[sl], [O.f64(v)[sl] for v in c["values"]], c["proj"], c["bases"],
                            c["w1s"], c["w2s"], G=w.G, H_kv=w.H_kv, d=w.d, n_res=w.n_res, coef_fmt=w.coef_fmt,
                            res_fmt=w.res_fmt, pos=None if c["pos"] is None else c["pos"][sl],
                            keys_post_rope=c["keys_post_rope"], theta=w.theta)


def _proj_abs_bound(c, sl):
    """Worst-case fp32 accumulation error of the projection per coefficient: N * 2^-24 * sum_n |k_n p_n|."""
    K = np.abs(O.f64(c["keys"])[sl]).reshape(-1, c["proj"].shape[1])
    P = np.abs(O.f64(c["proj"]))
    N = P.shape[1]
    return (K @ P.T).reshape(O.f64(c["keys"])[sl].shape[:2] + (P.shape[0],)) * N * 2.0 ** -24


def _proj_err_band(c, sl):
    """Width of the band around a bf16 rounding boundary inside which a float32 projection may round differently
    from the fp64 one: 16 sqrt(N) 2^-24 sqrt(sum_n (k_n p_n)^2) per coefficient.  The rounding errors of an N-term
    float32 sum add like a random walk whose standard deviation is about 2^-24 sqrt(N/6) sqrt(sum_n (k_n p_n)^2),
    so the band is about 39 of them wide on each side; a float32 emulation of the projection at these shapes flips
    ~0.04 % of the coefficients, all inside it (and the band holds ~4 % of them)."""
    K = O.f64(c["keys"])[sl].reshape(-1, c["proj"].shape[1])
    P = O.f64(c["proj"])
    N = P.shape[1]
    sq = np.sqrt((K * K) @ (P * P).T)
    return (16.0 * np.sqrt(N) * 2.0 ** -24 * sq).reshape(O.f64(c["keys"])[sl].shape[:2] + (P.shape[0],))


def exact_projection_case(w: synth.Workload) -> dict:
    """A write-side case with no rounding decision to flip: bf16 keys (not low rank) and a 0/1 selection `proj`
    that copies r of the G*H_kv*d stacked key features into the coefficients, with the bases its exact inverse
    (proj . stacked bases = I).  Each coefficient is then one key feature times 1 plus zeros, exact in float32 and
    fp64 alike, so the stored coefficients must equal the oracle's bit for bit and the residual index sets may
    differ only within 1e-3 of the cut-off.  Values are the predictor of the true keys plus noise, so the rebuilt
    keys (the selected features, zeros elsewhere) predict them with errors spread over a wide range."""
    assert w.act == "bf16" and w.coef_fmt == "bf16"
    D = w.G * w.H_kv * w.d
    keys = synth.gaussian((w.B, w.T, w.G, w.H_kv, w.d), 1.0, w.seed, w.name, "exact-keys", 0).to(torch.bfloat16)
    gen = torch.Generator().manual_seed(synth.sub_seed(w.seed, w.name, 0, "exact-subset"))
    idx = torch.sort(torch.randperm(D, generator=gen)[: w.r]).values
    proj = torch.zeros((w.r, D), dtype=torch.float32)
    proj[torch.arange(w.r), idx] = 1.0
    W_stack = proj.T.contiguous()                                  # [D, r]: W_stack[idx[k], k] = 1
    rows = w.H_kv * w.d
    bases = [W_stack[l * rows:(l + 1) * rows].to(torch.bfloat16).contiguous() for l in range(w.G)]
    raw = synth.draw_group(w, 0, with_noise=True)
    k64 = O.f64(keys)
    values = [torch.from_numpy(O.predict_values(k64[:, :, l], raw["w1"][l], raw["w2"][l]) +
                               O.f64(raw["noise"][l])).to(torch.bfloat16) for l in range(w.G)]
    return dict(w=w, keys=keys, values=values, proj=proj, bases=bases, w1s=raw["w1"], w2s=raw["w2"], pos=None,
                keys_post_rope=False, coef_raw_draw=None)


# Bounds on the rows whose stored coefficients differ between the float32 GPU projection and the fp64 one.  A bf16
# coefficient flips with probability ~4e-4 (float32 emulation), so a row of r <= 640 flips with probability up
# to ~1 - (1 - 4e-4)^640 = 23 %; an int4 group flips only where a quotient or a scale sits on a rounding tie, and
# a flipped fp16 group scale changes all 32 coefficients of its group (at most ~one group per flipped row:
# 0.05 of the rows x 32 / 512 coefficients = 3.1e-3).
FLIP_ROWS_MAX = {"bf16": 0.35, "int4": 0.05, "f32": 0.0}
FLIP_COEF_MAX = {"bf16": 2e-3, "int4": 4e-3, "f32": 0.0}


def check_compress(gpu: dict, orc: dict, w: synth.Workload, c: dict, bs=None):
    """Stored coefficients are valid roundings of the oracle's unrounded projection (within the fp32
    accumulation bound); errors, residual index sets and residual rows match.

    A bf16 coefficient may differ from the oracle's rounding only where the oracle's unrounded value lies within
    the float32 error band (_proj_err_band) of a bf16 rounding boundary; int4 and bf16 flips are counted, printed
    and bounded (FLIP_ROWS_MAX, FLIP_COEF_MAX).  A token whose stored coefficients came out differently on the
    two sides gets a different error, so it may enter or leave the residual set on either side; what is unique
    is the ranking of the other tokens: the GPU's residual tokens outside that flipped set must be the oracle's
    top ones among the unflipped tokens, up to the 1e-3 band at that cut-off."""
    sl = slice(None) if bs is None else bs
    raw = orc["coef_raw"]
    acc = _proj_abs_bound(c, sl)
    stats = {}
    if w.coef_fmt == "int4":
        g_codes = gpu["coef"].cpu()[sl].numpy()
        g_scale = gpu["coef_scale"].cpu()[sl].double().numpy()
        g_vals = O.dequant_int4_g32(g_codes, g_scale)
        s_full = np.repeat(g_scale, 32, axis=-1)
        assert np.all(np.abs(g_vals - raw) <= s_full / 2 * (1 + 1e-3) + acc + 1e-7), "int4 codes are not a valid rounding"
        o_scale = orc["coef_scale"]
        assert np.all(np.abs(g_scale - o_scale) <= np.abs(o_scale) * 2.0 ** -10 + 1e-12)
        flipped_rows = np.any(g_codes != orc["coef_q"], axis=-1) | np.any(g_scale != o_scale, axis=-1)   # [B, T]
        stats["flipped_coef_frac"] = float(np.mean(g_vals != orc["coef"]))
    else:
        g_vals = gpu["coef"].cpu()[sl].double().numpy()
        if w.coef_fmt == "bf16":
            assert np.all(np.abs(g_vals - raw) <= np.abs(raw) * 2.0 ** -8 + acc * (1 + 2.0 ** -8) + 1e-12), \
                "bf16 coefficients misrounded"
        else:
            assert np.all(np.abs(g_vals - raw) <= np.abs(raw) * 2.0 ** -24 + acc + 1e-12)
        # float32 storage has no rounding decision to flip; 16-bit storage flips where the fp32 and fp64
        # projections straddle a rounding boundary
        flipped = (g_vals != orc["coef"]) if w.coef_fmt == "bf16" else np.zeros(g_vals.shape, bool)
        flipped_rows = np.any(flipped, axis=-1)
        stats["flipped_coef_frac"] = float(flipped.mean())
        if flipped.any():
            # only coefficients whose unrounded value is within the float32 error band of a rounding boundary
            band = _proj_err_band(c, sl)
            lo, hi = O.round_bf16(raw - band), O.round_bf16(raw + band)
            outside = flipped & (lo == hi)
            assert not outside.any(), \
                f"{int(outside.sum())} bf16 coefficients differ from the oracle's rounding away from any boundary"
    stats["flipped_row_frac"] = float(flipped_rows.mean())
    print(f"compress parity: {stats['flipped_coef_frac']:.2e} of the stored coefficients and "
          f"{stats['flipped_row_frac']:.3f} of the token rows differ from the oracle's rounding")
    assert stats["flipped_coef_frac"] <= FLIP_COEF_MAX[w.coef_fmt], stats
    assert stats["flipped_row_frac"] <= FLIP_ROWS_MAX[w.coef_fmt], stats
    B, T = flipped_rows.shape
    for l in range(w.G):
        lay = orc["layers"][l]
        g_err = gpu["err"][l].cpu()[sl].double().numpy()             # [B, H_kv, T]
        same = ~flipped_rows[:, None, :].repeat(w.H_kv, 1)
        ed = np.abs(g_err - lay["err"])[same]
        stats[f"err_maxdiff_l{l}"] = float(ed.max()) if ed.size else 0.0
        assert ed.size == 0 or float(ed.max()) <= 1e-4, f"layer {l}: err differs by {float(ed.max()):.3g}"
        if w.n_res == 0:
            continue
        g_idx = gpu["res_idx"][l].cpu()[sl].numpy()
        for b in range(B):
            F = set(np.nonzero(flipped_rows[b])[0].tolist())
            for h in range(w.H_kv):
                gs = g_idx[b, h].tolist()
                assert gs == sorted(set(gs)), f"layer {l} (b={b}, h={h}): residual list not strictly ascending"
                g_rest = set(gs) - F
                n_rest = len(g_rest)
                e = lay["err"][b, h]
                order = sorted((t for t in range(T) if t not in F), key=lambda t: (-e[t], t))
                want = set(order[:n_rest])
                if n_rest == 0 or g_rest == want:
                    continue
                cut = e[order[n_rest - 1]]
                for t in g_rest ^ want:
                    assert abs(e[t] - cut) <= BAND, \
                        f"layer {l} (b={b}, h={h}): token {t} differs, {abs(e[t] - cut):.3g} from the cut-off"
        # residual rows of tokens kept by both sides, with unflipped coefficients
        if w.res_fmt == "int8":
            g_rv = O.dequant_int8_vec(gpu["res_val"][l].cpu()[sl].numpy(), gpu["res_scale"][l].cpu()[sl].double().numpy())
        else:
            g_rv = gpu["res_val"][l].cpu()[sl].double().numpy()
        o_rv = lay["res_val"]
        for b in range(B):
            for h in range(w.H_kv):
                gi = {t: j for j, t in enumerate(g_idx[b, h].tolist())}
                for j, t in enumerate(lay["res_idx"][b, h].tolist()):
                    if t in gi and not flipped_rows[b, t]:
                        gv, ov = g_rv[b, h, gi[t]], o_rv[b, h, j]
                        tol = (np.abs(ov).max() / 127.0 + 1e-4) if w.res_fmt == "int8" else (np.abs(ov) * 2.0 ** -7 + 1e-4)
                        assert np.all(np.abs(gv - ov) <= tol), f"layer {l} (b={b}, h={h}) residual row of token {t}"
    print("compress parity:", stats)
    return stats

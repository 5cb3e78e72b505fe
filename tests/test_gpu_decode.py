"""GPU parity of lowram_decode_attn against the fp64 oracle, through the C ABI.

Small cases (the oracle runs the whole problem) span several tiles with ragged tails for every workload
shape; full-size cases run the GPU at the benchmark's sizes and compare sampled (sequence, kv-head) pairs
that the oracle recomputes independently.  Edge cases: empty inputs, S >= T (selection is a no-op), S = 1,
no residuals, every token a residual, exact ties, and the device check word on bad indices.
"""
import numpy as np
import pytest
import torch

import lowram_cases as C
import oracle as O
from decode_attention_19_b300 import synth

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

SMALL = {
    "tiny": W["tiny"],
    "tiny_ragged_S": W["tiny"].with_(T=250, S=100),
    "llama8b_small": W["llama8b"].with_(B=2, T=1000, S=300),
    "long_small": W["long"].with_(B=1, T=1500, S=400),
    "peak_small": W["peak"].with_(B=3, T=777, S=200),
    "evict_quant_small": W["evict_quant"].with_(B=2, T=3000, T_nominal=12000, S=500),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_bf16_and_int4_workloads_take_the_tensor_core_key_pass():
    import decode_attention_19_b300 as L
    for name in ["llama8b", "long", "peak"]:
        w = W[name]
        sh = L.lowram_decode_shape(w.B, w.T, w.H_q, w.H_kv, w.d, w.r, w.m, w.S, w.n_res, 1, 1, 1, w.T, 0.0)
        assert L.lowram_decode_uses_tensor_cores(sh), name
    tiny = W["tiny"]
    sh = L.lowram_decode_shape(1, 256, 4, 2, 64, 32, 64, 256, 64, 0, 0, 0, 256, 0.0)
    assert not L.lowram_decode_uses_tensor_cores(sh)
    # int4 coefficients with bf16 activations: an fp16 copy (or the exact two-term bf16 split of rank 2r), then
    # the same kernels
    w = W["evict_quant"]
    sh = L.lowram_decode_shape(w.B, w.T, w.H_q, w.H_kv, w.d, w.r, w.m, w.S, w.n_res, 1, 2, 3, w.T_nominal, 0.0)
    assert L.lowram_decode_uses_tensor_cores(sh)
    sh.flags = L.FLAG_INT4_EXACT_SPLIT
    assert L.lowram_decode_uses_tensor_cores(sh)
    sh = L.lowram_decode_shape(w.B, w.T, w.H_q, w.H_kv, w.d, 1024, w.m, w.S, w.n_res, 1, 2, 3, w.T_nominal, 0.0)
    assert L.lowram_decode_uses_tensor_cores(sh)        # fp16 copy of rank 1024
    sh.flags = L.FLAG_INT4_EXACT_SPLIT
    assert not L.lowram_decode_uses_tensor_cores(sh)   # rank 2r = 2048 is past the key pass's limit


def test_rope_table_matches_fp64_angles():
    import decode_attention_19_b300 as L
    for d, theta, n in [(64, 1e4, 300), (128, 5e5, 65536)]:
        cos, sin = L.lowram_rope_table(d, theta, n)
        cos, sin = cos.cpu().double().numpy(), sin.cpu().double().numpy()
        for p in [0, 1, 17, n // 2, n - 1]:
            c, s = O.rope_angles(d, theta, p)
            np.testing.assert_allclose(cos[:, p], c, atol=1e-7, rtol=0)
            np.testing.assert_allclose(sin[:, p], s, atol=1e-7, rtol=0)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("biases", [False, True])
def test_decode_small_matches_oracle(name, biases):
    w = SMALL[name]
    c = C.decode_case(w, biases=biases)
    gpu = C.run_gpu_decode(c)
    orc = C.run_oracle_decode(c)
    C.check_decode(gpu, orc, w.S_eff)


@pytest.mark.parametrize("H_q,H_kv,r", [(8, 8, 512), (6, 3, 256), (16, 2, 512), (4, 1, 384), (7, 1, 128),
                                         (32, 8, 1024), (14, 2, 640)])
def test_decode_head_ratios_and_ranks(H_q, H_kv, r):
    """Every q-heads-per-kv-head ratio of the key pass, one and two kv-heads per unit (odd H_kv takes one),
    the resident-latent and streamed feeding modes (r = 640 and 1024 stream)."""
    w = SMALL["llama8b_small"].with_(B=2, T=700, S=200, H_q=H_q, H_kv=H_kv, r=r)
    c = C.decode_case(w)
    C.check_decode(C.run_gpu_decode(c), C.run_oracle_decode(c), w.S_eff)


@pytest.mark.parametrize("S", [0, 1, 7, 129, 999, 1000, 5000])
def test_decode_selection_sizes(S):
    w = SMALL["llama8b_small"].with_(S=S)
    c = C.decode_case(w)
    gpu = C.run_gpu_decode(c, S=S)
    orc = C.run_oracle_decode(c, S=S)
    S_eff = min(S, w.T)
    C.check_decode(gpu, orc, S_eff)
    if S_eff == 0:
        assert np.all(gpu["out"] == 0) and np.all(np.isneginf(gpu["lse"]))


@pytest.mark.parametrize("rho", [0.0, 1.0])
def test_decode_residual_extremes(rho):
    w = SMALL["llama8b_small"].with_(rho=rho)
    c = C.decode_case(w)
    if rho == 0.0:
        assert c["res_idx"].shape[-1] == 0
    C.check_decode(C.run_gpu_decode(c), C.run_oracle_decode(c), w.S_eff)


@pytest.mark.parametrize("T", [1, 31, 33, 127, 129])
def test_decode_tiny_token_counts(T):
    w = SMALL["llama8b_small"].with_(T=T, S=min(T, 17))
    c = C.decode_case(w)
    C.check_decode(C.run_gpu_decode(c), C.run_oracle_decode(c), w.S_eff)


def test_decode_exact_ties_take_the_lower_index():
    w = SMALL["llama8b_small"].with_(B=1, T=300, S=100)
    c = C.decode_case(w)
    # copy token 10's latents and position onto tokens 11..40: identical keys in every head
    coef = c["coef"].clone()
    coef[0, 11:41] = coef[0, 10]
    c["coef"] = coef
    c["coef_vals"] = O.f64(coef)
    pos = torch.arange(w.T, dtype=torch.int32)[None].clone()
    pos[0, 11:41] = 10
    c["pos"] = pos
    gpu = C.run_gpu_decode(c)
    orc = C.run_oracle_decode(c)
    assert np.array_equal(gpu["key"][0, :, 10:41], np.repeat(gpu["key"][0, :, 10:11], 31, axis=1))
    C.check_decode(gpu, orc, w.S_eff)
    # where the cut falls inside the tie block the lower indices are kept: the kept members of the block
    # form a prefix of it
    for h in range(w.H_kv):
        kept = [t for t in gpu["sel"][0, h] if 10 <= t <= 40]
        assert kept == list(range(10, 10 + len(kept)))


def test_decode_ties_across_the_cluster_split():
    # a row long enough to be split over a cluster of two CTAs (8192 keys each, the second partly filled), a
    # block of equal keys straddling the split, and S chosen so that kv-head 0's cut falls inside the block
    w = SMALL["llama8b_small"].with_(B=1, T=12000, S=100)
    c = C.decode_case(w)
    t0, t1 = 8180, 8206
    coef = c["coef"].clone()
    coef[0, t0 + 1:t1] = coef[0, t0]
    c["coef"] = coef
    c["coef_vals"] = O.f64(coef)
    pos = torch.arange(w.T, dtype=torch.int32)[None].clone()
    pos[0, t0 + 1:t1] = t0
    c["pos"] = pos
    probe = C.run_gpu_decode(c)
    k0 = probe["key"][0, 0]
    assert np.all(k0[t0:t1] == k0[t0])
    S = int((k0 > k0[t0]).sum()) + 20
    gpu = C.run_gpu_decode(c, S=S)
    orc = C.run_oracle_decode(c, S=S)
    C.check_decode(gpu, orc, S)
    kept = [int(t) for t in gpu["sel"][0, 0] if t0 <= t < t1]
    assert kept == list(range(t0, t0 + 20))
    assert np.all(np.diff(gpu["sel"][0], axis=-1) > 0)


def test_decode_empty_batch_and_empty_cache():
    import decode_attention_19_b300 as L
    w = SMALL["llama8b_small"].with_(T=0, S=10, rho=0.0)
    c = C.decode_case(w)
    gpu = C.run_gpu_decode(c, hooks=False)
    assert np.all(gpu["out"] == 0) and np.all(np.isneginf(gpu["lse"]))
    w0 = SMALL["llama8b_small"].with_(B=0)
    c0 = C.decode_case(w0)
    gpu0 = C.run_gpu_decode(c0, hooks=False)
    assert gpu0["out"].shape == (0, w.H_q, w.d)


def test_device_check_word_flags_bad_residual_list_and_positions():
    import decode_attention_19_b300 as L
    w = SMALL["llama8b_small"]
    c = C.decode_case(w)
    ws = torch.zeros(1 << 24, dtype=torch.uint8, device="cuda")
    C.run_gpu_decode(c, workspace=ws)
    assert L.lowram_get_error(ws) == 0
    bad = c["res_idx"].clone()
    bad[0, 0, 5] = bad[0, 0, 4]          # not strictly ascending (still in range)
    c2 = dict(c, res_idx=bad)
    C.run_gpu_decode(c2, workspace=ws)
    assert L.lowram_get_error(ws) & L.CHECK_RES_INDEX
    assert L.lowram_get_error(ws) == 0   # cleared by the read
    pos = torch.arange(w.T, dtype=torch.int32)[None].repeat(w.B, 1)
    pos[1, 7] = 5000                     # beyond the tables (max_pos = T): clamped and flagged
    c3 = dict(c, pos=pos)
    C.run_gpu_decode(c3, workspace=ws)
    assert L.lowram_get_error(ws) & L.CHECK_POS_RANGE


FULL = ["tiny", "llama8b", "long", "peak", "evict_quant"]


@pytest.mark.parametrize("name", FULL)
def test_decode_full_size_sampled(name):
    """The benchmark's sizes on the GPU; the oracle recomputes sampled (sequence, kv-head) sub-problems."""
    w = W[name]
    c = C.decode_case(w)
    gpu = C.run_gpu_decode(c)
    g = w.H_q // w.H_kv
    samples = [(0, 0), (w.B - 1, w.H_kv - 1)] if w.B * w.H_kv > 1 else [(0, 0)]
    for b, h in samples:
        sub = C.slice_case(c, [b], [h])
        orc = C.run_oracle_decode(sub)
        part = {"out": gpu["out"][b:b + 1, h * g:(h + 1) * g], "lse": gpu["lse"][b:b + 1, h * g:(h + 1) * g],
                "key": gpu["key"][b:b + 1, h:h + 1], "sel": gpu["sel"][b:b + 1, h:h + 1]}
        C.check_decode(part, orc, w.S_eff)


def _per_sequence(c, per_basis, per_mlp):
    """Sequence b gets layer b's basis and/or predictor (with biases) of the same draw: different weights per
    sequence, stacked along a leading batch dimension."""
    w = c["w"]
    raw = synth.draw_group(w.with_(G=max(w.G, w.B)), 0, with_noise=False)
    c = dict(c)
    act = c["w1"].dtype
    if per_basis:
        c["basis"] = torch.stack([raw["basis"][b] for b in range(w.B)]).to(act)
    if per_mlp:
        c["w1"] = torch.stack([raw["w1"][b] for b in range(w.B)]).to(act)
        c["w2"] = torch.stack([raw["w2"][b] for b in range(w.B)]).to(act)
        c["b1"] = synth.gaussian((w.B, w.H_kv, w.m), 0.1, w.seed, w.name, "b1-seq", 0)
        c["b2"] = synth.gaussian((w.B, w.H_kv, w.d), 0.1, w.seed, w.name, "b2-seq", 0)
    return c


@pytest.mark.parametrize("name,per_basis,per_mlp", [
    ("llama8b_small", True, False), ("llama8b_small", False, True), ("llama8b_small", True, True),
    ("peak_small", True, True), ("tiny_ragged_S", True, True), ("evict_quant_small", True, True)])
def test_decode_per_sequence_bases_and_predictors(name, per_basis, per_mlp):
    """A basis and a predictor per sequence (the batch strides of the C shape): each sequence is decoded with its
    own weights.  peak_small has an odd number of 128-token tiles per sequence, so the key pass's tile pairs must
    stay inside a sequence; the int4 workload runs with a repeated basis per sequence."""
    w = SMALL[name].with_(B=3)
    c = _per_sequence(C.decode_case(w), per_basis, per_mlp)
    C.check_decode(C.run_gpu_decode(c), C.run_oracle_decode(c), w.S_eff)


@pytest.mark.parametrize("exact", [False, True])
@pytest.mark.parametrize("H_q,H_kv,r", [(32, 8, 512), (28, 4, 384), (16, 2, 1024)])
def test_decode_int4_fp16_copy_and_exact_split(exact, H_q, H_kv, r):
    """int4 caches on the tensor cores: the default fp16 copy of code * scale (keys within KEY_TOL_INT4_F16) and
    the exact two-term bf16 split (keys within KEY_TOL); r = 1024 takes the fp16 copy only."""
    if exact and r > 512:
        pytest.skip("the exact split doubles the rank past the key pass's limit")
    w = SMALL["evict_quant_small"].with_(H_q=H_q, H_kv=H_kv, r=r)
    c = C.decode_case(w)
    C.check_decode(C.run_gpu_decode(c, int4_exact_split=exact), C.run_oracle_decode(c), w.S_eff)

"""GPU parity of lowram_compress (the write side) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import lowram_cases as C
from decode_attention_19_b300 import synth

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS

SMALL = {
    "tiny": W["tiny"],
    "llama8b_small": W["llama8b"].with_(B=2, T=1000),
    "long_small": W["long"].with_(B=1, T=1100),
    "peak_small": W["peak"].with_(B=2, T=777),
    "evict_quant_small": W["evict_quant"].with_(B=2, T=3000, T_nominal=12000),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("name", list(SMALL))
def test_compress_small_matches_oracle(name):
    w = SMALL[name]
    c = C.compress_case(w)
    C.check_compress(C.run_gpu_compress(c), C.run_oracle_compress(c), w, c)


@pytest.mark.parametrize("name", ["llama8b_small", "evict_quant_small"])
def test_compress_keys_given_after_rope(name):
    w = SMALL[name]
    c = C.compress_case(w, keys_post_rope=True)
    C.check_compress(C.run_gpu_compress(c), C.run_oracle_compress(c), w, c)


@pytest.mark.parametrize("name", ["llama8b_small", "peak_small"])
def test_compress_exact_projection_has_no_exemptions(name):
    """With a 0/1 selection projection nothing can round differently: every stored coefficient equals the oracle's
    (and the selected key feature) bit for bit, and the residual index sets match the oracle's except within 1e-3
    of the cut-off, with no token exempt."""
    w = SMALL[name]
    c = C.exact_projection_case(w)
    gpu = C.run_gpu_compress(c)
    orc = C.run_oracle_compress(c)
    stats = C.check_compress(gpu, orc, w, c)
    assert stats["flipped_coef_frac"] == 0.0 and stats["flipped_row_frac"] == 0.0
    sel = c["proj"].argmax(dim=1)
    want = c["keys"].reshape(w.B, w.T, -1)[:, :, sel]
    assert torch.equal(gpu["coef"].cpu(), want)


@pytest.mark.parametrize("rho", [0.0, 1.0])
def test_compress_residual_extremes(rho):
    w = SMALL["llama8b_small"].with_(rho=rho)
    c = C.compress_case(w)
    gpu = C.run_gpu_compress(c)
    C.check_compress(gpu, C.run_oracle_compress(c), w, c)
    if rho == 1.0:
        assert all(np.array_equal(gpu["res_idx"][l].cpu().numpy()[b, h], np.arange(w.T))
                   for l in range(w.G) for b in range(w.B) for h in range(w.H_kv))


@pytest.mark.parametrize("name", ["llama8b", "evict_quant"])
def test_compress_full_size_sampled(name):
    """Full-size write side on the GPU; the oracle recomputes one sequence (sequences are independent)."""
    w = W[name]
    c = C.compress_case(w)
    gpu = C.run_gpu_compress(c)
    b = [w.B - 1]
    C.check_compress(gpu, C.run_oracle_compress(c, bs=b), w, c, bs=b)


def _decode_inputs(w, l, coef, coef_vals, res_idx, res_val, res_vals64, basis, w1, w2):
    return dict(w=w, coef=coef, coef_vals=coef_vals, coef_scale=None, basis=basis, w1=w1, w2=w2,
                q=synth.draw_query(w, l), res_idx=res_idx, res_val=res_val, res_vals64=res_vals64, res_scale=None,
                pos=None, b1=None, b2=None, max_pos=w.T)


# Each chain rounds its own latents: where the fp32 projection and the fp64 one fall on opposite sides of a bf16
# rounding boundary, a stored coefficient differs by one bf16 step (check_compress bounds these), which moves a
# rebuilt key by up to ~1e-3; selections are still compared exactly outside the cut-off band.
CHAIN_KEY_TOL = 2e-3


def test_compress_then_decode_round_trip():
    """A cache written by lowram_compress decodes like the oracle's decode of the oracle's own compressed cache
    (each side runs its whole chain; nothing crosses from the GPU to the oracle)."""
    import oracle as O
    w = SMALL["llama8b_small"]
    c = C.compress_case(w)
    gpu = C.run_gpu_compress(c)
    orc = C.run_oracle_compress(c)
    for l in [0, w.G - 1]:
        dg = _decode_inputs(w, l, gpu["coef"].cpu(), None, gpu["res_idx"][l].cpu(), gpu["res_val"][l].cpu(), None,
                            c["bases"][l], c["w1s"][l], c["w2s"][l])
        lay = orc["layers"][l]
        do = _decode_inputs(w, l, None, orc["coef"], lay["res_idx"], None, lay["res_val"], c["bases"][l],
                            c["w1s"][l], c["w2s"][l])
        C.check_decode(C.run_gpu_decode(dg), C.run_oracle_decode(do), w.S_eff, key_tol=CHAIN_KEY_TOL)


def test_fit_compress_decode_chain():
    """Prompt keys -> fitted cross-layer basis -> compress -> decode on the GPU, against the oracle's own chain
    (eigendecomposition, compress, decode).  The two fitted bases differ by a rotation inside the same subspace,
    so the latents differ while the rebuilt keys and the decode outputs agree; float32 activations keep the
    stored bases exact enough for index-set parity."""
    import decode_attention_19_b300 as L
    import oracle as O
    w = W["tiny"].with_(B=2, T=300, S=120)
    c = C.compress_case(w)
    proj_g, bases_g, ws = L.lowram_fit_basis(c["keys"].cuda(), w.r, iters=8, seed=7)
    torch.cuda.synchronize()
    assert L.lowram_get_error(ws) == 0
    proj_o, bases_o, _ = O.fit_basis(c["keys"], w.r, w.G, w.H_kv, w.d)
    cg = dict(c, proj=proj_g.cpu(), bases=[b.cpu() for b in bases_g])
    co = dict(c, proj=torch.as_tensor(proj_o, dtype=torch.float32),
              bases=[torch.as_tensor(b, dtype=torch.float32) for b in bases_o])
    gpu = C.run_gpu_compress(cg)
    orc = C.run_oracle_compress(co)
    for l in range(w.G):
        dg = _decode_inputs(w, l, gpu["coef"].cpu(), None, gpu["res_idx"][l].cpu(), gpu["res_val"][l].cpu(), None,
                            cg["bases"][l], c["w1s"][l], c["w2s"][l])
        lay = orc["layers"][l]
        do = _decode_inputs(w, l, None, orc["coef"], lay["res_idx"], None, lay["res_val"], co["bases"][l],
                            c["w1s"][l], c["w2s"][l])
        C.check_decode(C.run_gpu_decode(dg), C.run_oracle_decode(do), w.S_eff, key_tol=CHAIN_KEY_TOL)

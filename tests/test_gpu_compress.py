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


def test_compress_then_decode_round_trip():
    """A cache written by lowram_compress decodes like the oracle's decode of the same stored cache."""
    import oracle as O
    w = SMALL["llama8b_small"]
    c = C.compress_case(w)
    gpu = C.run_gpu_compress(c)
    for l in [0, w.G - 1]:
        d = dict(w=w, coef=gpu["coef"].cpu(), coef_vals=O.f64(gpu["coef"].cpu()), coef_scale=None,
                 basis=c["bases"][l], w1=c["w1s"][l], w2=c["w2s"][l], q=synth.draw_query(w, l),
                 res_idx=gpu["res_idx"][l].cpu(), res_val=gpu["res_val"][l].cpu(),
                 res_vals64=O.f64(gpu["res_val"][l].cpu()), res_scale=None, pos=None, b1=None, b2=None,
                 max_pos=w.T)
        C.check_decode(C.run_gpu_decode(d), C.run_oracle_decode(d), w.S_eff)

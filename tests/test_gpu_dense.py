"""GPU parity of the uncompressed-cache comparator (lowram_dense_decode_attn) against the fp64 oracle.

The comparator is the same kernel family on an explicit, already rotated K/V cache [B, T, H_kv, d]; it is what
the compressed cache replaces.  Cases span several split ranges and a ragged tail, every supported q-heads per
kv-head ratio, both head dims, bf16 and float32 storage, and the empty cache.
"""
import numpy as np
import pytest
import torch

import oracle as O
from decode_attention_19_b300 import synth

pytestmark = pytest.mark.gpu

OUT_MAX_ABS = 1e-2
OUT_REL_L2 = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _case(B, T, H_q, H_kv, d, dtype, seed):
    dt = {"bf16": "bf16", "f32": "f32"}[dtype]
    q = synth.gaussian((B, H_q, d), d ** -0.5, seed, "dense-q", dtype=dt)
    k = synth.gaussian((B, T, H_kv, d), 1.0, seed, "dense-k", dtype=dt)
    v = synth.gaussian((B, T, H_kv, d), 1.0, seed, "dense-v", dtype=dt)
    return q, k, v


@pytest.mark.parametrize("B,T,H_q,H_kv,d,dtype", [
    (2, 1000, 32, 8, 128, "bf16"),    # llama-shaped heads, ragged tail
    (1, 4097, 28, 4, 128, "bf16"),    # seven queries per kv-head
    (3, 777, 8, 8, 64, "bf16"),       # one query per kv-head, d = 64
    (2, 300, 16, 8, 64, "f32"),
    (1, 5, 8, 1, 128, "f32"),         # fewer tokens than one warp step
    (1, 2049, 16, 2, 128, "bf16"),    # eight queries per kv-head
])
def test_dense_matches_oracle(B, T, H_q, H_kv, d, dtype):
    import decode_attention_19_b300 as L
    q, k, v = _case(B, T, H_q, H_kv, d, dtype, 3)
    out, lse = L.lowram_dense_decode_attn(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    ref_out, ref_lse = O.dense_decode(q, k, v)
    got = out.cpu().double().numpy()
    err = np.abs(got - ref_out).max()
    rel = np.linalg.norm(got - ref_out) / np.linalg.norm(ref_out)
    assert err <= OUT_MAX_ABS and rel <= OUT_REL_L2, (err, rel)
    np.testing.assert_allclose(lse.cpu().double().numpy(), ref_lse, atol=1e-3, rtol=0)


def test_dense_full_size_sampled():
    """The benchmark's comparator shape (B=8, T=8192, H_q=32, H_kv=8); the oracle recomputes two sequences."""
    import decode_attention_19_b300 as L
    q, k, v = _case(8, 8192, 32, 8, 128, "bf16", 5)
    out, lse = L.lowram_dense_decode_attn(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    for b in (0, 7):
        ref_out, ref_lse = O.dense_decode(q[b:b + 1], k[b:b + 1], v[b:b + 1])
        got = out[b:b + 1].cpu().double().numpy()
        assert np.abs(got - ref_out).max() <= OUT_MAX_ABS
        assert np.linalg.norm(got - ref_out) / np.linalg.norm(ref_out) <= OUT_REL_L2
        np.testing.assert_allclose(lse[b:b + 1].cpu().double().numpy(), ref_lse, atol=1e-3, rtol=0)


def test_dense_empty_cache():
    import decode_attention_19_b300 as L
    q, k, v = _case(2, 0, 8, 2, 64, "bf16", 1)
    out, lse = L.lowram_dense_decode_attn(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert np.all(out.cpu().numpy() == 0) and np.all(np.isneginf(lse.cpu().numpy()))

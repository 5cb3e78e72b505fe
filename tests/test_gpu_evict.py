"""GPU parity of the heavy-hitter eviction plan: the attention mass of an observation window over the prompt's
tokens (against the oracle's fp64 softmax sums; bf16 prompts take the tensor-core path, float32 ones the CUDA
cores), and the kept tokens (exact index sets: sinks, recents, the heaviest others, ties to the lower index).
Shapes: several q-heads per kv-head ratios, both head dims, bf16 and float32, ragged token tiles, windows of 1 to
40 queries, long prompts with several token tiles per CTA.
"""
import numpy as np
import pytest
import torch

import lowram_cases as C
import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def window_case(B, T, W, H_q, H_kv, d, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn((B, W, H_q, d), generator=g) * 2 * d ** -0.5).to(dtype)
    k = torch.randn((B, T, H_kv, d), generator=g).to(dtype)
    return q, k


@pytest.mark.parametrize("B,T,W,H_q,H_kv,d,dtype", [
    (2, 1000, 32, 32, 8, 128, torch.bfloat16),
    (1, 777, 4, 28, 4, 128, torch.bfloat16),
    (2, 300, 1, 16, 2, 64, torch.float32),
    (3, 65, 8, 8, 8, 64, torch.bfloat16),
    (1, 160013, 2, 4, 1, 64, torch.bfloat16),    # long prompt: several token tiles per CTA, ragged tail
    (1, 160013, 2, 4, 1, 64, torch.float32),
    (2, 4000, 40, 8, 1, 128, torch.bfloat16),    # 320 window query-heads per kv-head: three query tiles
])
def test_attention_mass_matches_oracle(B, T, W, H_q, H_kv, d, dtype):
    import decode_attention_19_b300 as L
    q, k = window_case(B, T, W, H_q, H_kv, d, dtype, 1)
    mass = L.lowram_attention_mass(q.cuda(), k.cuda())
    torch.cuda.synchronize()
    got = O.f64(mass.cpu())
    ref = O.attention_mass(q, k)
    np.testing.assert_allclose(got, ref, rtol=2e-4, atol=1e-6 * W * H_q)
    np.testing.assert_allclose(got.sum(axis=1), W * H_q, rtol=1e-4)


@pytest.mark.parametrize("T,n_sink,n_recent,T_keep", [(1000, 64, 100, 400), (333, 3, 30, 33), (50, 4, 6, 50)])
def test_evict_plan_matches_oracle_exactly(T, n_sink, n_recent, T_keep):
    import decode_attention_19_b300 as L
    rng = np.random.default_rng(2)
    mass = rng.random((3, T)).astype(np.float32)
    mass[1, 100:140] = 0.75                              # a block of ties across the cut
    keep = L.lowram_evict_plan(torch.as_tensor(mass).cuda(), n_sink=n_sink, n_recent=n_recent, T_keep=T_keep)
    torch.cuda.synchronize()
    assert np.array_equal(keep.cpu().numpy(), O.evict_plan(mass, n_sink, n_recent, T_keep))


def test_window_mass_to_plan_chain():
    """GPU mass -> GPU plan against the oracle's mass -> plan: kept sets equal except within 1e-4 (relative) of the
    cut-off mass."""
    import decode_attention_19_b300 as L
    B, T, W, H_q, H_kv, d = 2, 2000, 16, 32, 8, 128
    q, k = window_case(B, T, W, H_q, H_kv, d, torch.bfloat16, 3)
    mass = L.lowram_attention_mass(q.cuda(), k.cuda())
    keep = L.lowram_evict_plan(mass, n_sink=16, n_recent=128, T_keep=500)
    torch.cuda.synchronize()
    ref_mass = O.attention_mass(q, k)
    ref = O.evict_plan(ref_mass, 16, 128, 500)
    scores = ref_mass.copy()                             # the forced tokens rank first
    scores[:, :16] = np.inf
    scores[:, T - 128:] = np.inf
    C.check_index_sets(keep.cpu().numpy(), ref, scores, 500, band=1e-4 * float(ref_mass.max()), what="kept tokens")

"""GPU parity of the fitted cross-layer key basis (lowram_fit_basis) against the fp64 oracle.

The GPU finds the top-r subspace by subspace iteration, the oracle by a full eigendecomposition, and any
orthonormal basis of the subspace serves the method; so the tests compare what is unique: the subspace (its
projector), the rebuild error of the keys against the optimal one, and proj . stacked bases = I.  Keys are
low-rank with a decaying spectrum plus noise (a clear gap after rank r), given pre-RoPE or rotated at scattered
positions, in float32 and bf16; keys of rank below r must raise the device check bit.
"""
import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def low_rank_keys(B, T, G, H_kv, d, r, noise, seed, dtype):
    rng = np.random.default_rng(seed)
    D = G * H_kv * d
    U, _ = np.linalg.qr(rng.normal(0, 1, (D, r)))
    C = rng.normal(0, 1, (B * T, r)) * np.geomspace(8.0, 1.0, r)
    K = (C @ U.T + noise * rng.normal(0, 1, (B * T, D))).reshape(B, T, G, H_kv, d)
    return torch.as_tensor(K, dtype=torch.float32).to(dtype)


def check_fit(proj, bases, keys, r, G, H_kv, d, dtype, **kw):
    K = O.f64(keys)
    B, T = K.shape[0], K.shape[1]
    po, _, _ = O.fit_basis(K, r, G, H_kv, d, **kw)
    pg = O.f64(proj)
    D = G * H_kv * d
    # subspace: projectors agree
    np.testing.assert_allclose(pg.T @ pg, po.T @ po, atol=2e-4)
    # proj is a left inverse of the stacked bases (bf16 bases: rounding of the basis entries)
    Wg = np.concatenate([O.f64(b) for b in bases], axis=0)
    np.testing.assert_allclose(pg @ Wg, np.eye(r), atol=1e-5 if dtype == torch.float32 else 1e-2)
    # rebuild error of the (RoPE-inverted) keys within 1e-3 of the optimal one
    if kw.get("keys_post_rope"):
        pos = np.broadcast_to(np.asarray(kw["pos"])[:, :, None, None], (B, T, G, H_kv))
        K = O.rope_rows(K, pos, kw["theta"], inverse=True)
    Kf = K.reshape(B * T, D)
    eg = np.linalg.norm(Kf - Kf @ pg.T @ pg)
    eo = np.linalg.norm(Kf - Kf @ po.T @ po)
    assert eg <= eo * (1 + 1e-3), (eg, eo)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("B,T,G,H_kv,d,r", [(2, 300, 2, 2, 64, 64), (1, 777, 4, 1, 128, 96), (3, 100, 1, 8, 64, 256),
                                             (1, 1500, 2, 4, 128, 640), (1, 600, 3, 6, 128, 64)])
def test_fit_basis_matches_oracle(dtype, B, T, G, H_kv, d, r):
    # D = 2304 (the last case): 90 Gram tiles, enough that each owns its outputs (stored, not added), as at full size
    import decode_attention_19_b300 as L
    keys = low_rank_keys(B, T, G, H_kv, d, r, 0.05, 1, dtype)
    proj, bases, ws = L.lowram_fit_basis(keys.cuda(), r, iters=8, seed=3)
    torch.cuda.synchronize()
    assert L.lowram_get_error(ws) == 0
    check_fit(proj, bases, keys, r, G, H_kv, d, dtype)


def test_fit_basis_inverts_rope():
    import decode_attention_19_b300 as L
    B, T, G, H_kv, d, r, theta = 2, 400, 2, 2, 64, 64, 1e4
    keys_pre = low_rank_keys(B, T, G, H_kv, d, r, 0.05, 2, torch.float32)
    rng = np.random.default_rng(5)
    pos = np.stack([np.sort(rng.choice(2000, T, replace=False)) for _ in range(B)]).astype(np.int32)
    P = np.broadcast_to(pos[:, :, None, None], (B, T, G, H_kv))
    keys = torch.as_tensor(O.rope_rows(O.f64(keys_pre), P, theta), dtype=torch.float32)
    cos, sin = L.lowram_rope_table(d, theta, 2000)
    proj, bases, ws = L.lowram_fit_basis(keys.cuda(), r, pos=torch.as_tensor(pos).cuda(), rope_cos=cos, rope_sin=sin,
                                         keys_post_rope=True, iters=8)
    torch.cuda.synchronize()
    assert L.lowram_get_error(ws) == 0
    check_fit(proj, bases, keys, r, G, H_kv, d, torch.float32, pos=pos, keys_post_rope=True, theta=theta)


def test_fit_basis_flags_keys_of_lower_rank():
    import decode_attention_19_b300 as L
    keys = low_rank_keys(2, 200, 2, 2, 64, 32, 0.0, 4, torch.float32)    # rank 32, asked for 64
    _, _, ws = L.lowram_fit_basis(keys.cuda(), 64, iters=4)
    torch.cuda.synchronize()
    assert L.lowram_get_error(ws) & L.CHECK_NOT_PD

"""GPU parity of the exact tail (tokens decoded after compression, kept as explicit rotated K and V) and of the
log-sum-exp merge of body and tail, through the C ABI, against the fp64 oracle.

Cases: rows appended one at a time land bit-exact in place and leave the other rows untouched; attention over
the first t_len rows of a strided tail buffer (every q-heads per kv-head ratio, both head dims, bf16 and float32,
t_len = 0); the merge with empty sets and in place; and a whole decode step -- compressed body plus a tail of
appended tokens -- against the oracle's body, tail and merge.
"""
import numpy as np
import pytest
import torch

import lowram_cases as C
import oracle as O
from decode_attention_19_b300 import synth

pytestmark = pytest.mark.gpu

OUT_MAX_ABS = 1e-2
OUT_REL_L2 = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_tail_append_writes_rows_in_place(dtype, d):
    import decode_attention_19_b300 as L
    B, T_cap, H_kv = 3, 7, 2
    g = torch.Generator().manual_seed(1)
    tk = torch.full((B, T_cap, H_kv, d), 7.0, dtype=dtype).cuda()
    tv = torch.full((B, T_cap, H_kv, d), -7.0, dtype=dtype).cuda()
    want_k, want_v = tk.cpu().clone(), tv.cpu().clone()
    for t in [0, 3, 6, 3]:
        kn = torch.randn((B, H_kv, d), generator=g).to(dtype)
        vn = torch.randn((B, H_kv, d), generator=g).to(dtype)
        L.lowram_tail_append(kn.cuda(), vn.cuda(), tk, tv, t)
        want_k[:, t], want_v[:, t] = kn, vn
    torch.cuda.synchronize()
    assert torch.equal(tk.cpu(), want_k) and torch.equal(tv.cpu(), want_v)
    with pytest.raises(L.LowramError):
        L.lowram_tail_append(kn.cuda(), vn.cuda(), tk, tv, T_cap)


@pytest.mark.parametrize("B,T_cap,t_len,H_q,H_kv,d,dtype", [
    (2, 64, 37, 32, 8, 128, torch.bfloat16),     # llama-shaped heads, ragged length inside the buffer
    (3, 300, 300, 28, 4, 128, torch.bfloat16),   # seven queries per kv-head, buffer full
    (2, 40, 1, 16, 2, 128, torch.bfloat16),      # eight queries per kv-head, one token
    (2, 50, 29, 8, 8, 64, torch.float32),
    (1, 16, 0, 8, 2, 64, torch.bfloat16),        # empty tail
])
def test_tail_attention_matches_oracle(B, T_cap, t_len, H_q, H_kv, d, dtype):
    import decode_attention_19_b300 as L
    g = torch.Generator().manual_seed(2)
    q = (torch.randn((B, H_q, d), generator=g) * d ** -0.5).to(dtype)
    tk = torch.randn((B, T_cap, H_kv, d), generator=g).to(dtype)
    tv = torch.randn((B, T_cap, H_kv, d), generator=g).to(dtype)
    out, lse = L.lowram_tail_decode_attn(q.cuda(), tk.cuda(), tv.cuda(), t_len)
    torch.cuda.synchronize()
    got, got_lse = out.cpu().double().numpy(), lse.cpu().double().numpy()
    if t_len == 0:
        assert np.all(got == 0) and np.all(np.isneginf(got_lse))
        return
    ref, ref_lse = O.dense_decode(q, tk[:, :t_len], tv[:, :t_len])
    C.check_out(got, ref, OUT_MAX_ABS, OUT_REL_L2)
    np.testing.assert_allclose(got_lse, ref_lse, atol=1e-3, rtol=0)


@pytest.mark.parametrize("in_place", [False, True])
def test_merge_matches_oracle(in_place):
    import decode_attention_19_b300 as L
    B, H_q, d = 4, 8, 128
    rng = np.random.default_rng(3)
    oa, ob = rng.normal(0, 1, (B, H_q, d)), rng.normal(0, 1, (B, H_q, d))
    la, lb = rng.normal(0, 3, (B, H_q)), rng.normal(0, 3, (B, H_q))
    la[0, :3] = -np.inf                      # body empty for some heads
    lb[1, :2] = -np.inf                      # tail empty for some heads
    la[2, 0] = lb[2, 0] = -np.inf            # both empty
    f = lambda x: torch.as_tensor(x, dtype=torch.float32).cuda()
    ta, tla, tb, tlb = f(oa), f(la), f(ob), f(lb)
    if in_place:
        out, lse = L.lowram_merge_attn(ta, tla, tb, tlb, out=ta, lse=tla)
    else:
        out, lse = L.lowram_merge_attn(ta, tla, tb, tlb)
    torch.cuda.synchronize()
    ref, ref_lse = O.merge_attn(O.round_f32(oa), O.round_f32(la), O.round_f32(ob), O.round_f32(lb))
    np.testing.assert_allclose(out.cpu().double().numpy(), ref, atol=2e-6, rtol=1e-5)
    got_lse = lse.cpu().double().numpy()
    assert np.array_equal(np.isneginf(got_lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], atol=1e-5, rtol=0)


@pytest.mark.parametrize("n_tail", [1, 9])
def test_decode_step_with_exact_tail_matches_oracle(n_tail):
    """Compressed body (lowram_decode_attn) + tail of n_tail appended tokens (lowram_tail_append, then
    lowram_tail_decode_attn) merged with lowram_merge_attn, against the oracle's decode, tail attention and merge."""
    import decode_attention_19_b300 as L
    w = synth.WORKLOADS["llama8b"].with_(B=2, T=1000, S=300)
    c = C.decode_case(w)
    body = C.run_gpu_decode(c, hooks=False)
    orc = C.run_oracle_decode(c)
    T_cap = 16
    g = torch.Generator().manual_seed(4)
    tk = torch.zeros((w.B, T_cap, w.H_kv, w.d), dtype=torch.bfloat16).cuda()
    tv = torch.zeros_like(tk)
    kt = (torch.randn((w.B, n_tail, w.H_kv, w.d), generator=g) * 4).to(torch.bfloat16)
    vt = torch.randn((w.B, n_tail, w.H_kv, w.d), generator=g).to(torch.bfloat16)
    for t in range(n_tail):
        L.lowram_tail_append(kt[:, t].contiguous().cuda(), vt[:, t].contiguous().cuda(), tk, tv, t)
    q = c["q"].cuda()
    o_tail, l_tail = L.lowram_tail_decode_attn(q, tk, tv, n_tail)
    out, lse = L.lowram_merge_attn(torch.as_tensor(body["out"], dtype=torch.float32).cuda(),
                                   torch.as_tensor(body["lse"], dtype=torch.float32).cuda(), o_tail, l_tail)
    torch.cuda.synchronize()
    ref_t, ref_tl = O.dense_decode(c["q"], kt, vt)
    ref, ref_lse = O.merge_attn(orc.out, orc.lse, ref_t, ref_tl)
    C.check_out(out.cpu().double().numpy(), ref, OUT_MAX_ABS, OUT_REL_L2)
    np.testing.assert_allclose(lse.cpu().double().numpy(), ref_lse, atol=1e-3, rtol=0)

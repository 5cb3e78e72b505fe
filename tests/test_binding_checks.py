"""The binding's buffer checks (CPU, no GPU needed).

The C entry points see raw pointers and the sizes the binding passes, so a tensor smaller than the layout its
call reads or writes would send a kernel outside the buffer.  The binding checks every tensor against those
sizes (element count and element size) before anything reaches the library; these cases must all be refused
with LowramShapeError (or TypeError for mixed dtypes) while the tensors are still on the host.
"""
import pytest
import torch

import decode_attention_19_b300 as L

bf, f32 = torch.bfloat16, torch.float32


def _decode_inputs(B=2, T=40, H_q=8, H_kv=2, d=64, r=64, m=32, n_res=4):
    return dict(q=torch.zeros(B, H_q, d, dtype=bf), coef=torch.zeros(B, T, r, dtype=bf),
                basis=torch.zeros(H_kv * d, r, dtype=bf), w1=torch.zeros(H_kv, m, d, dtype=bf),
                w2=torch.zeros(H_kv, d, m, dtype=bf), rope_cos=torch.zeros(d // 2, T, dtype=f32),
                rope_sin=torch.zeros(d // 2, T, dtype=f32), res_idx=torch.zeros(B, H_kv, n_res, dtype=torch.int32),
                res_val=torch.zeros(B, H_kv, n_res, d, dtype=bf))


def _decode(x, **over):
    x = dict(x, **over)
    return L.lowram_decode_attn(x.pop("q"), x.pop("coef"), x.pop("basis"), x.pop("w1"), x.pop("w2"), S=8, **x)


@pytest.mark.parametrize("name,bad", [
    ("basis", torch.zeros(2 * 64, 32, dtype=bf)),              # rank 32 against a rank-64 cache
    ("w2", torch.zeros(2, 64, 32, dtype=f32)),                 # float32 weights with bf16 activations
    ("rope_sin", torch.zeros(32, 20, dtype=f32)),              # shorter table than the cosines
    ("res_val", torch.zeros(2, 2, 3, 64, dtype=bf)),           # fewer rows than residual indices
    ("pos", torch.zeros(2, 39, dtype=torch.int32)),            # one position short
    ("b1", torch.zeros(2, 16, dtype=f32)),                     # half the hidden width
    ("out", torch.zeros(2, 8, 32, dtype=f32)),                 # half the head dim
    ("sel_out", torch.zeros(2, 2, 7, dtype=torch.int32)),      # fewer slots than min(S, T) = 8
])
def test_decode_refuses_undersized_or_mistyped_buffers(name, bad):
    with pytest.raises(L.LowramShapeError, match=name):
        _decode(_decode_inputs(), **{name: bad})


def test_decode_int4_needs_its_scales():
    x = _decode_inputs()
    x["coef"] = torch.zeros(2, 40, 32, dtype=torch.uint8)     # int4 codes for rank 64
    with pytest.raises(L.LowramShapeError, match="coef_scale"):
        _decode(x)
    with pytest.raises(L.LowramShapeError, match="coef_scale"):
        _decode(x, coef_scale=torch.zeros(2, 40, 1, dtype=torch.float16))


def test_static_decode_refuses_a_missing_or_small_output():
    x = _decode_inputs()
    args = [x.pop(k) for k in ("q", "coef", "basis", "w1", "w2")]
    with pytest.raises(L.LowramShapeError, match="out"):
        L.lowram_decode_attn_static(*args, S=8, out=None, **x)
    with pytest.raises(L.LowramShapeError, match="lse"):
        L.lowram_decode_attn_static(*args, S=8, out=torch.zeros(2, 8, 64), lse=torch.zeros(2, 7), **x)


def test_compress_checks_every_layer_of_the_group():
    B, T, G, H_kv, d, r, m = 1, 16, 2, 2, 64, 64, 32
    keys = torch.zeros(B, T, G, H_kv, d, dtype=bf)
    ok = dict(values=[torch.zeros(B, T, H_kv, d, dtype=bf)] * G, proj=torch.zeros(r, G * H_kv * d, dtype=f32),
              bases=[torch.zeros(H_kv * d, r, dtype=bf)] * G, w1s=[torch.zeros(H_kv, m, d, dtype=bf)] * G,
              w2s=[torch.zeros(H_kv, d, m, dtype=bf)] * G)

    def call(**over):
        a = dict(ok, **over)
        return L.lowram_compress(keys, a["values"], a["proj"], a["bases"], a["w1s"], a["w2s"], n_res=2,
                                 coef_dtype=L.LOWRAM_BF16, res_dtype=L.LOWRAM_BF16)
    with pytest.raises(L.LowramShapeError, match="values"):
        call(values=ok["values"][:1])                          # one layer's values missing
    with pytest.raises(L.LowramShapeError, match="w2s"):
        call(w2s=[ok["w2s"][0], torch.zeros(H_kv, d, 16, dtype=bf)])
    with pytest.raises(L.LowramShapeError, match="proj"):
        call(proj=torch.zeros(r, G * H_kv * d, dtype=torch.float16))


def test_dense_tail_merge_and_mass_refuse_mismatched_buffers():
    q = torch.zeros(2, 8, 64, dtype=bf)
    k = torch.zeros(2, 30, 2, 64, dtype=bf)
    with pytest.raises(L.LowramShapeError, match="v"):
        L.lowram_dense_decode_attn(q, k, torch.zeros(2, 29, 2, 64, dtype=bf))
    with pytest.raises(L.LowramShapeError, match="k"):
        L.lowram_dense_decode_attn(torch.zeros(3, 8, 64, dtype=bf), k, k)      # a third sequence K does not hold
    with pytest.raises(L.LowramShapeError, match="tail_v"):
        L.lowram_tail_decode_attn(q, k, torch.zeros(2, 20, 2, 64, dtype=bf), 10)
    oa, la = torch.zeros(2, 8, 64), torch.zeros(2, 8)
    with pytest.raises(L.LowramShapeError, match="out_b"):
        L.lowram_merge_attn(oa, la, torch.zeros(2, 8, 32), la)
    with pytest.raises(TypeError):
        L.lowram_attention_mass(torch.zeros(2, 4, 8, 64, dtype=f32), k)
    with pytest.raises(L.LowramShapeError, match="k"):
        L.lowram_attention_mass(torch.zeros(2, 4, 8, 128, dtype=bf), k)       # head dim 128 against 64


class _OnDevice:
    """Stand-in for a contiguous CUDA tensor on device `idx` (the check reads only these attributes)."""

    def __init__(self, idx):
        self.is_cuda = True
        self.device = torch.device("cuda", idx)

    def is_contiguous(self):
        return True


def test_every_tensor_of_a_call_must_share_one_device():
    from decode_attention_19_b300 import binding as B
    assert B._dev(_OnDevice(1), None, _OnDevice(1)) == torch.device("cuda", 1)
    with pytest.raises(L.LowramShapeError, match="one device"):
        B._dev(_OnDevice(0), _OnDevice(1))


def test_batch_strides_follow_the_weight_ranks():
    x = _decode_inputs(B=3)
    shared = L.decode_shape(x["q"], x["coef"], x["w1"], S=8, n_res=4, max_pos=40, res_dtype=1, basis=x["basis"])
    assert shared.basis_batch_stride == 0 and shared.mlp_batch_stride == 0
    basis = torch.zeros(3, 2 * 64, 64, dtype=bf)
    w1 = torch.zeros(3, 2, 32, 64, dtype=bf)
    sh = L.decode_shape(x["q"], x["coef"], w1, S=8, n_res=4, max_pos=40, res_dtype=1, basis=basis)
    assert sh.basis_batch_stride == 2 * 64 * 64 and sh.mlp_batch_stride == 2 * 32 * 64
    assert (sh.H_kv, sh.m) == (2, 32)


def test_per_sequence_weights_must_cover_every_sequence():
    x = _decode_inputs(B=3)
    with pytest.raises(L.LowramShapeError, match="w2"):
        _decode(x, w1=torch.zeros(3, 2, 32, 64, dtype=bf), w2=torch.zeros(2, 2, 64, 32, dtype=bf))
    with pytest.raises(L.LowramShapeError, match="b1"):
        _decode(x, w1=torch.zeros(3, 2, 32, 64, dtype=bf), w2=torch.zeros(3, 2, 64, 32, dtype=bf),
                b1=torch.zeros(2, 32, dtype=f32))

"""lowram_decode_attn_static: the decode entry point for callers that cannot allocate device memory (code
inside another runtime's memory pool, plug-ins without an allocator, paths that must not allocate after
setup).  Its scratch is the library's static device array instead of a caller workspace.  It runs the same
kernels on the same inputs as lowram_decode_attn, whose reductions have a fixed order, so its results must be
bit-identical to that call's, call after call.

This file is named to be collected last, so a run that stops at the first failure has run everything else.
"""
import ctypes

import pytest
import torch

import lowram_cases as C
from decode_attention_19_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _inputs(w, layer):
    c = C.decode_case(w, layer=layer)
    dev = torch.device("cuda")
    cu = lambda t: None if t is None else t.to(dev).contiguous()
    return {k: cu(c[k]) for k in ("q", "coef", "basis", "w1", "w2", "res_idx", "res_val")}


def test_static_scratch_matches_workspace_call_twice_in_a_row():
    import decode_attention_19_b300 as L
    w = synth.WORKLOADS["llama8b"].with_(B=2, T=1000, S=300)
    cos, sin = L.lowram_rope_table(w.d, w.theta, w.T)
    for layer in (0, 1):                       # two calls in a row, on different inputs
        x = _inputs(w, layer)
        ref, ref_lse = L.lowram_decode_attn(x["q"], x["coef"], x["basis"], x["w1"], x["w2"], rope_cos=cos,
                                            rope_sin=sin, S=w.S, res_idx=x["res_idx"], res_val=x["res_val"])
        out = torch.empty_like(ref)
        lse = torch.empty_like(ref_lse)
        L.lowram_decode_attn_static(x["q"], x["coef"], x["basis"], x["w1"], x["w2"], rope_cos=cos, rope_sin=sin,
                                    S=w.S, res_idx=x["res_idx"], res_val=x["res_val"], out=out, lse=lse)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"layer {layer}: outputs differ by {float((out - ref).abs().max()):.3g}"
        assert torch.equal(lse, ref_lse)
        assert L.lowram_decode_attn_static_get_error() == 0     # clean inputs leave the check word clear


def test_static_scratch_rejects_shapes_beyond_its_size():
    import decode_attention_19_b300 as L
    # 256 sequences x 4 kv-heads x 32768 tokens of selection keys alone need 128 MiB of scratch
    sh = L.lowram_decode_shape(256, 32768, 28, 4, 128, 384, 128, 512, 3277, 1, 1, 1, 32768, 0.0)
    assert L.lowram_decode_workspace_size(sh) > (32 << 20)
    lib = L.lib()
    # every tensor pointer NULL: the size check answers first, and were it ever to pass, the NULL query would be
    # refused on the host before any launch
    st = lib.lowram_decode_attn_static(ctypes.byref(sh), *([None] * 18), None)
    assert st == 4
    assert "32 MiB" in lib.lowram_last_error().decode()

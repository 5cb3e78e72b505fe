"""Failure detection on the GPU without a fault: the tensor-core value pass bounds every pipeline wait, and a
call whose wait gives up returns with LOWRAM_CHECK_TIMEOUT in its check word while the context stays usable.

lowram_set_wait_limit shortens the limit to one SM cycle, so waits that would complete (a TMA stage landing,
the MMAs finishing) give up; the kernel then drains the copies and MMAs it issued, frees its tensor memory and
returns.  Nothing waits on a flag that is never set, nothing traps, and the next call with the default limit
must match the oracle."""
import pytest
import torch

import lowram_cases as C
from decode_attention_19_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_value_pass_wait_limit_expires_then_the_next_call_is_exact():
    import decode_attention_19_b300 as L
    w = synth.WORKLOADS["llama8b"].with_(B=2, T=1000, S=300)
    c = C.decode_case(w)
    ws = torch.zeros(1 << 26, dtype=torch.uint8, device="cuda")
    L.lowram_set_wait_limit(1)
    try:
        C.run_gpu_decode(c, workspace=ws)
        torch.cuda.synchronize()
        word = L.lowram_get_error(ws)
    finally:
        L.lowram_set_wait_limit(0)
    assert word & L.CHECK_TIMEOUT, f"check word {word:#x}: no wait gave up"
    gpu = C.run_gpu_decode(c, workspace=ws)
    assert L.lowram_get_error(ws) == 0
    C.check_decode(gpu, C.run_oracle_decode(c), w.S_eff)


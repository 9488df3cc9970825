"""The prefill's failure path, made to run on purpose and on the GPU without a fault.

Every wait of the chunked prefill is bounded. Here one unit's hand-off flag is withheld (a
test setting of the library, sala_gla_debug_prefill_knobs) and the wait for a predecessor's
state is limited to 1 ms, so the successor's wait gives up: the call must still return,
SALA_ERR_TIMEOUT must be recorded in the device status word, and the next ordinary call must
give correct results, which it cannot unless the aborted kernel drained its copies and MMAs
and released its tensor memory. Nothing faults or hangs: the wait that gives up is a bounded
poll of a flag in global memory.
"""
import time

import pytest
import torch

import oracle
from gated_linear_attention_gb300 import inputs

pytestmark = pytest.mark.gpu

SALA_ERR_TIMEOUT = 5


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_linear_attention_gb300 import build, sala_gla
    build.build()
    return sala_gla


def _case():
    # one sequence of 2048 tokens, 2 heads: segments of 640 tokens, so units (segment s, head h)
    # = 2 s + h; withholding unit 0 starves unit 2, and then unit 4 and unit 6 (head 0)
    w = inputs.Workload("fault", "prefill", H=2, seqlens=(2048,), qk_norm="l2",
                        gate="logsigmoid", h0=True, seed=41)
    return inputs.make_prefill(w)


def _run(sg, x):
    dev = torch.device("cuda")
    o, hT = sg.chunk_fwd(x["q"].to(dev), x["k"].to(dev), x["v"].to(dev), x["g"].to(dev),
                         x["scale"], h0=x["h0"].to(dev))
    return o, hT


def test_withheld_hand_off_times_out_then_next_call_is_correct(sg):
    x = _case()
    assert sg.get_device_status() == 0
    try:
        sg.debug_prefill_knobs(flag_wait_ns=1_000_000, withhold_unit=0)
        t0 = time.perf_counter()
        _run(sg, x)
        status = sg.get_device_status()          # synchronises
        dt = time.perf_counter() - t0
    finally:
        sg.debug_prefill_knobs()
    assert status == SALA_ERR_TIMEOUT
    assert dt < 1.0                              # three 1 ms waits gave up, not the 2 s default
    assert sg.get_device_status() == 0           # the status word was cleared by the read
    # the same problem again, normally: correct results
    o, hT = _run(sg, x)
    torch.cuda.synchronize()
    assert sg.get_device_status() == 0
    o_ref, h_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"], h0=x["h0"])
    assert oracle.rel_fro(o.cpu().float().reshape(o_ref.shape), o_ref) <= 1e-2
    assert oracle.rel_fro(hT.cpu(), h_ref) <= 5e-3


def test_knobs_reject_bad_unit(sg):
    with pytest.raises(sg.SalaError):
        sg.debug_prefill_knobs(0, -2)

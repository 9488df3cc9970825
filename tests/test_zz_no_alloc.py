"""The prefill entry point that allocates nothing (sala_gla_chunk_fwd_noalloc).

It serves callers that cannot allocate device memory while they run the layer: engines that
reserve nearly all of HBM for their own pools at start-up, plug-in hosts whose execute path
forbids allocation, and latency-critical loops that cannot afford an allocator call. Its
scratch is a fixed 64 MiB device array inside the library, shared by every call.

These tests call it through the C ABI and compare it with sala_gla_chunk_fwd (same
tolerances as the oracle parity tests: relative Frobenius error <= 1e-2 on o, <= 5e-3 on hT)
on two calls in a row with different shapes, so that anything left in the shared array by
the first call would show up in the second. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import oracle
from gated_linear_attention_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_linear_attention_gb300 import build, sala_gla
    build.build()
    return sala_gla.load()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call(fn, x, o, hT):
    q, k, v, g = (x[n].cuda() for n in ("q", "k", "v", "g"))
    h0 = None if x["h0"] is None else x["h0"].cuda()
    cu = None if x["cu_seqlens"] is None else x["cu_seqlens"].cuda()
    if cu is None:
        B, T, H = q.shape[0], q.shape[1], q.shape[2]
        nseq = 0
    else:
        B, T, H = 1, q.shape[0], q.shape[1]
        nseq = cu.numel() - 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(_p(q), _p(k), _p(v), _p(g), ctypes.c_float(x["scale"]), _p(h0), _p(cu), _p(o),
            _p(hT), B, T, H, nseq, stream)
    torch.cuda.synchronize()
    return rc


def _outputs(x):
    nseq = 1 if x["cu_seqlens"] is None else x["cu_seqlens"].numel() - 1
    if x["cu_seqlens"] is None:
        nseq = x["q"].shape[0]
    H = x["q"].shape[-2]
    o = torch.full(tuple(x["q"].shape), float("nan"), dtype=torch.bfloat16, device="cuda")
    hT = torch.full((nseq, H, 128, 128), float("nan"), device="cuda")
    return o, hT


CASES = [
    lambda: inputs.make_prefill("sala_layer"),
    lambda: inputs.make_prefill("varlen", seqlens=(0, 700, 1, 4096, 333)),
]


def test_noalloc_matches_allocating_entry_point_on_two_calls(lib):
    for make in CASES:                       # two calls in a row, different shapes
        x = make()
        o_ref, h_ref = _outputs(x)
        assert _call(lib.sala_gla_chunk_fwd, x, o_ref, h_ref) == 0
        o, hT = _outputs(x)
        assert _call(lib.sala_gla_chunk_fwd_noalloc, x, o, hT) == 0
        assert oracle.rel_fro(o.cpu().float(), o_ref.cpu().float()) <= 1e-2
        assert oracle.rel_fro(hT.cpu(), h_ref.cpu()) <= 5e-3
    from gated_linear_attention_gb300 import sala_gla
    assert sala_gla.get_device_status() == 0


def test_noalloc_lengthens_segments_to_fit_its_scratch(lib):
    # 28 sequences x 2048 tokens x 32 heads: the allocating path cuts 1024-token segments
    # (56 per head, 1792 units of 64 KB: 117 MB of hand-off states), which does not fit the
    # 64 MiB array; the no-alloc path lengthens the segments until at most ~1000 units remain
    # (here: one segment per sequence). The results agree within the parity tolerances.
    x = inputs.make_prefill("varlen", seqlens=(2048,) * 28, seed=17)
    o_ref, h_ref = _outputs(x)
    assert _call(lib.sala_gla_chunk_fwd, x, o_ref, h_ref) == 0
    o, hT = _outputs(x)
    assert _call(lib.sala_gla_chunk_fwd_noalloc, x, o, hT) == 0
    assert oracle.rel_fro(o.cpu().float(), o_ref.cpu().float()) <= 1e-2
    assert oracle.rel_fro(hT.cpu(), h_ref.cpu()) <= 5e-3
    from gated_linear_attention_gb300 import sala_gla
    assert sala_gla.get_device_status() == 0


def test_noalloc_repeated_call_is_stable(lib):
    x = inputs.make_prefill("tiny")
    o1, h1 = _outputs(x)
    o2, h2 = _outputs(x)
    assert _call(lib.sala_gla_chunk_fwd_noalloc, x, o1, h1) == 0
    assert _call(lib.sala_gla_chunk_fwd_noalloc, x, o2, h2) == 0
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_noalloc_rejects_problems_beyond_its_scratch(lib):
    # 64 sequences x 32 heads need more than 64 MiB of per-segment states: refused up front
    n, H = 64, 32
    q = torch.zeros((n, H, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.zeros((n, H), device="cuda")
    cu = torch.arange(n + 1, dtype=torch.int64, device="cuda")
    o = torch.empty_like(q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.sala_gla_chunk_fwd_noalloc(_p(q), _p(q), _p(q), _p(g), ctypes.c_float(0.1), None,
                                        _p(cu), _p(o), None, 1, n, H, n, stream)
    assert rc == 7                           # SALA_ERR_TOO_LARGE
    assert b"scratch" in lib.sala_gla_status_string(7)

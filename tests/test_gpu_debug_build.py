"""The debug build (compiled with SALA_GLA_DEBUG): device code checks the indices it derives
from the inputs and records SALA_ERR_DEBUG_CHECK instead of making a bad access. On valid
inputs it must give the oracle's results with a clean status word; on an input the release
build does not validate on the device (a q/k prologue's cu_seqlens that is not monotone, which
is still in bounds for the release kernel) it must report the check and leave the tokens it
could not place untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_attention_gb300 import inputs

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
S_TOL = 5e-3
DEBUG_CHECK = 9   # SALA_ERR_DEBUG_CHECK


@pytest.fixture(scope="module")
def dbg():
    """The binding with the debug library swapped in for this module's tests."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_linear_attention_gb300 import build, sala_gla
    build.build()
    release = sala_gla.load()
    debug = sala_gla.load(build.build(debug=True))
    sala_gla._lib = debug
    sala_gla.get_device_status()   # clear the debug library's status word
    yield sala_gla
    sala_gla._lib = release


def test_debug_prefill_varlen_matches_oracle(dbg):
    x = inputs.make_prefill("varlen", seqlens=(0, 5, 1, 64, 0, 130, 700), H=3, seed=5)
    o, hT = dbg.chunk_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["g"].cuda(), x["scale"],
                          h0=x["h0"].cuda(), cu_seqlens=x["cu_seqlens"].cuda())
    torch.cuda.synchronize()
    assert dbg.get_device_status() == 0
    o_ref, h_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"], h0=x["h0"],
                                    cu_seqlens=x["cu_seqlens"])
    assert oracle.rel_fro(o.cpu().float().reshape(o_ref.shape), o_ref) <= O_TOL
    assert oracle.rel_fro(hT.cpu(), h_ref) <= S_TOL


def test_debug_prefill_tiny_matches_oracle(dbg):
    x = inputs.make_prefill("tiny")
    o, hT = dbg.chunk_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["g"].cuda(), x["scale"])
    torch.cuda.synchronize()
    assert dbg.get_device_status() == 0
    o_ref, h_ref = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"])
    assert oracle.rel_fro(o.cpu().float().reshape(o_ref.shape), o_ref) <= O_TOL
    assert oracle.rel_fro(hT.cpu(), h_ref) <= S_TOL


def test_debug_gdn_chunked_matches_oracle(dbg):
    x = inputs.make_prefill("varlen", seqlens=(200, 63, 129), H=2, seed=9)
    beta = torch.sigmoid(torch.randn(x["g"].shape, generator=torch.Generator().manual_seed(9)))
    o, hT = dbg.gdn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["g"].cuda(), beta.cuda(),
                        x["scale"], h0=x["h0"].cuda(), cu_seqlens=x["cu_seqlens"].cuda(),
                        chunked=True)
    torch.cuda.synchronize()
    assert dbg.get_device_status() == 0
    o_ref, h_ref = oracle.gdn_recurrent(x["q"], x["k"], x["v"], x["g"], beta, x["scale"],
                                        h0=x["h0"], cu_seqlens=x["cu_seqlens"])
    assert oracle.rel_fro(o.cpu().float().reshape(o_ref.shape), o_ref) <= O_TOL
    assert oracle.rel_fro(hT.cpu(), h_ref) <= S_TOL


def _prologue_inputs(T, H, seed):
    gen = torch.Generator().manual_seed(seed)
    q = (3 * torch.randn((T, H, 128), generator=gen)).to(torch.bfloat16)
    k = (3 * torch.randn((T, H, 128), generator=gen)).to(torch.bfloat16)
    qw = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    return q, k, qw, kw


def test_debug_prologue_valid_matches_oracle(dbg):
    q, k, qw, kw = _prologue_inputs(150, 4, seed=3)
    cu = torch.tensor([0, 70, 150], dtype=torch.int64)
    qd, kd = q.cuda(), k.cuda()
    dbg.qk_prologue(qd, kd, qw.cuda(), kw.cuda(), 1e-6, 10000.0, cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    assert dbg.get_device_status() == 0
    pos = np.concatenate([np.arange(70), np.arange(80)])
    assert oracle.rel_fro(qd.cpu().float(), oracle.qk_prologue(q, qw, pos[:, None])) <= 5e-3
    assert oracle.rel_fro(kd.cpu().float(), oracle.qk_prologue(k, kw, pos[:, None])) <= 5e-3


def test_debug_prologue_reports_unplaceable_tokens(dbg):
    # cu_seqlens [0, 80, 90, 50] over 100 tokens: the search places tokens 90-99 in sequence 2,
    # which ends at 50 (the release kernel stays in bounds and rotates them by tok - 90); the
    # debug build reports the check and leaves those tokens as they were
    q, k, qw, kw = _prologue_inputs(100, 2, seed=4)
    cu = torch.tensor([0, 80, 90, 50], dtype=torch.int64)
    qd, kd = q.cuda(), k.cuda()
    dbg.qk_prologue(qd, kd, qw.cuda(), kw.cuda(), 1e-6, 10000.0, cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    assert dbg.get_device_status() == DEBUG_CHECK
    assert dbg.get_device_status() == 0   # reading the word clears it
    assert torch.equal(qd.cpu()[90:], q[90:]) and torch.equal(kd.cpu()[90:], k[90:])
    pos = np.arange(80)
    assert oracle.rel_fro(qd.cpu()[:80].float(), oracle.qk_prologue(q[:80], qw, pos[:, None])) <= 5e-3


def test_debug_pooled_decode_matches_oracle(dbg):
    d = inputs.make_decode_steps("decode", 0, 1, nseq=6, H=3)
    p = inputs.make_decode_pool(nseq=6, H=3, pool=10, storage="f32", pad=(1,))
    pool = p["pool"].cuda()
    o = dbg.recurrent_step_indexed(d["q"][0].cuda(), d["k"][0].cuda(), d["v"][0].cuda(),
                                   d["g"][0].cuda(), d["scale"], pool, p["indices"].cuda())
    torch.cuda.synchronize()
    assert dbg.get_device_status() == 0
    idx = p["indices"]
    live = [n for n in range(6) if int(idx[n]) >= 0]
    S0 = p["pool"][idx[live]]
    cu = torch.arange(len(live) + 1, dtype=torch.int64)
    o_ref, S_ref = oracle.recurrent(d["q"][0][live], d["k"][0][live], d["v"][0][live],
                                    d["g"][0][live], d["scale"], h0=S0, cu_seqlens=cu)
    assert oracle.rel_fro(o.cpu().float()[live], o_ref) <= O_TOL
    assert oracle.rel_fro(pool.cpu()[idx[live]], S_ref) <= S_TOL

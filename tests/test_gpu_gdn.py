"""Parity of the gated-delta-rule decode step (sala_gla_gdn_recurrent_step, through the C ABI)
with the fp64 oracle's recurrence: relative Frobenius <= 1e-2 on o and <= 5e-3 on the states."""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_attention_gb300 import inputs

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
S_TOL = 5e-3


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_linear_attention_gb300 import build, sala_gla
    build.build()
    return sala_gla


def _run(sg, N, H, steps, w="gdn_decode"):
    x = inputs.make_decode_steps(w, 0, steps, nseq=N, H=H)
    beta = inputs.make_gdn_beta(w, 0, steps, nseq=N, H=H)
    S0 = inputs.make_decode_state(w, nseq=N, H=H)
    S = S0.cuda().clone()
    outs = []
    for s in range(steps):
        outs.append(sg.gdn_recurrent_step(x["q"][s].cuda(), x["k"][s].cuda(), x["v"][s].cuda(),
                                          x["g"][s].cuda(), beta[s].cuda(), x["scale"], S).cpu())
    torch.cuda.synchronize()
    return x, beta, S0, torch.stack(outs), S.cpu()


def _ref(x, beta, S0, seqs, steps):
    N, H = len(seqs), x["q"].shape[2]
    sel = lambda t: t[:steps, seqs].transpose(0, 1).reshape(N * steps, *t.shape[2:]).contiguous()
    cu = torch.arange(N + 1, dtype=torch.int64) * steps
    return oracle.gdn_recurrent(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["g"]), sel(beta),
                                x["scale"], h0=S0[seqs], cu_seqlens=cu)


@pytest.mark.parametrize("N,H,steps", [(1, 1, 1), (5, 3, 9), (16, 32, 4)])
def test_gdn_decode_small(sg, N, H, steps):
    x, beta, S0, od, S = _run(sg, N, H, steps)
    o_ref, h_ref = _ref(x, beta, S0, list(range(N)), steps)
    assert oracle.rel_fro(od.transpose(0, 1).reshape(N * steps, H, 128).float(), o_ref) <= O_TOL
    assert oracle.rel_fro(S, h_ref) <= S_TOL


def test_gdn_decode_steps_equal_chunked_form(sg):
    # the GPU recurrence over 70 steps equals the oracle's chunked (UT transform) form
    N, H, steps = 2, 4, 70
    x, beta, S0, od, S = _run(sg, N, H, steps)
    sel = lambda t: t.transpose(0, 1).reshape(N * steps, *t.shape[2:]).contiguous()
    cu = torch.arange(N + 1, dtype=torch.int64) * steps
    o_ref, h_ref = oracle.gdn_chunkwise(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["g"]), sel(beta),
                                        x["scale"], h0=S0, cu_seqlens=cu, chunk=64)
    assert oracle.rel_fro(sel(od).float(), o_ref) <= O_TOL
    assert oracle.rel_fro(S, h_ref) <= S_TOL


def test_gdn_full_size_sampled(sg):
    # the benchmark's configuration (256 sequences x 32 heads), 100 steps, 4 sequences checked
    w = inputs.WORKLOADS["gdn_decode"]
    steps = 100
    x, beta, S0, od, S = _run(sg, w.nseq, w.H, steps)
    seqs = [0, 63, 128, 255]
    o_ref, h_ref = _ref(x, beta, S0, seqs, steps)
    N = len(seqs)
    assert oracle.rel_fro(od[:, seqs].transpose(0, 1).reshape(N * steps, w.H, 128).float(), o_ref) <= O_TOL
    assert oracle.rel_fro(S[seqs], h_ref) <= S_TOL

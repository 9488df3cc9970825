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


# ---------------------------------------------------------------------------------------
# the recurrent form over whole sequences (sala_gla_gdn_fwd)


def _gdn_prefill_inputs(lens, H, seed):
    x = inputs.make_prefill("varlen", seqlens=tuple(lens), H=H, seed=seed)
    gen = torch.Generator().manual_seed(seed)
    beta = torch.sigmoid(torch.randn(x["g"].shape, generator=gen))
    return x, beta


@pytest.mark.parametrize("lens", [[1], [5, 0, 130, 64], [700, 300]])
def test_gdn_prefill_packed(sg, lens):
    x, beta = _gdn_prefill_inputs(lens, 4, seed=sum(lens))
    cu = x["cu_seqlens"]
    o, hT = sg.gdn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["g"].cuda(), beta.cuda(),
                       x["scale"], h0=x["h0"].cuda(), cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.gdn_chunkwise(x["q"], x["k"], x["v"], x["g"], beta, x["scale"],
                                        h0=x["h0"], cu_seqlens=cu)
    assert oracle.rel_fro(o.cpu().float(), o_ref) <= O_TOL
    assert oracle.rel_fro(hT.cpu(), h_ref) <= S_TOL
    for n, L in enumerate(lens):                 # an empty sequence returns h0
        if L == 0:
            assert torch.equal(hT[n].cpu(), x["h0"][n])


def test_gdn_prefill_rows_without_state(sg):
    x, beta = _gdn_prefill_inputs([96] * 3, 2, seed=21)
    q, k, v = (x[n].reshape(3, 96, 2, 128) for n in ("q", "k", "v"))
    g, b = x["g"].reshape(3, 96, 2), beta.reshape(3, 96, 2)
    o, hT = sg.gdn_fwd(q.cuda(), k.cuda(), v.cuda(), g.cuda(), b.cuda(), x["scale"])
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.gdn_recurrent(q, k, v, g, b, x["scale"])
    assert oracle.rel_fro(o.cpu().float().reshape(o_ref.shape), o_ref) <= O_TOL
    assert oracle.rel_fro(hT.cpu(), h_ref) <= S_TOL


def test_gdn_prefill_then_decode_equals_longer_prefill(sg):
    # prefill 50 tokens, then 10 decode steps from its final state == prefill of 60 tokens
    x, beta = _gdn_prefill_inputs([60], 3, seed=33)
    q, k, v, g = (x[n].cuda() for n in ("q", "k", "v", "g"))
    b, cu = beta.cuda(), torch.tensor([0, 50], dtype=torch.int64, device="cuda")
    o1, h1 = sg.gdn_fwd(q[:50].contiguous(), k[:50].contiguous(), v[:50].contiguous(), g[:50].contiguous(),
                        b[:50].contiguous(), x["scale"], h0=x["h0"].cuda(), cu_seqlens=cu)
    outs = []
    for t in range(50, 60):
        # (fresh copies: a row of g or beta alone is not 16-byte aligned for 3 heads)
        outs.append(sg.gdn_recurrent_step(q[t:t + 1].clone(), k[t:t + 1].clone(),
                                          v[t:t + 1].clone(), g[t:t + 1].clone(),
                                          b[t:t + 1].clone(), x["scale"], h1))
    o_all, h_all = sg.gdn_fwd(q, k, v, g, b, x["scale"], h0=x["h0"].cuda(),
                              cu_seqlens=torch.tensor([0, 60], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    od = torch.cat([o1] + outs)
    assert oracle.rel_fro(od.cpu().float(), o_all.cpu().float()) <= 5e-3
    assert oracle.rel_fro(h1.cpu(), h_all.cpu()) <= 1e-5


def test_gdn_prefill_gates_leaving_the_range(sg):
    # a gate of exactly 0 (g = -inf), single gates far below 2^-40, a run of strong decay and
    # gates above 1: the kernel keeps the running product of the gates apart from the state
    # and folds it in whenever it leaves [2^-40, 2^40]; the direct recurrence is the reference
    x, beta = _gdn_prefill_inputs([200, 90], 2, seed=41)
    g = x["g"].clone()
    g[10] = float("-inf")
    g[50, 0] = -60.0
    g[100:140] = -3.0
    g[150:160] = 0.7
    g[230] = -200.0
    cu = x["cu_seqlens"]
    o, hT = sg.gdn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), g.cuda(), beta.cuda(),
                       x["scale"], h0=x["h0"].cuda(), cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    o_ref, h_ref = oracle.gdn_recurrent(x["q"], x["k"], x["v"], g, beta, x["scale"],
                                        h0=x["h0"], cu_seqlens=cu)
    assert torch.isfinite(o.cpu().float()).all() and torch.isfinite(hT.cpu()).all()
    assert oracle.rel_fro(o.cpu().float(), o_ref) <= O_TOL
    assert oracle.rel_fro(hT.cpu(), h_ref) <= S_TOL
    # the output right after the zero gate sees only that token's own write
    o10 = oracle.gdn_recurrent(x["q"][10:11], x["k"][10:11], x["v"][10:11], g[10:11],
                               beta[10:11], x["scale"],
                               cu_seqlens=torch.tensor([0, 1], dtype=torch.int64))[0]
    assert oracle.rel_fro(o[10:11].cpu().float(), o10) <= O_TOL


def test_gdn_prefill_bench_size_sampled(sg):
    # the recurrent prefill at the benchmark's size and launch (64 sequences x 256 tokens,
    # 32 heads, inputs as the benchmark draws them); three sequences checked against the oracle
    lens = (256,) * 64
    x = inputs.make_prefill("varlen", seqlens=lens, H=32, seed=13)
    beta = torch.sigmoid(torch.randn(x["g"].shape, generator=torch.Generator().manual_seed(13)))
    o, hT = sg.gdn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["g"].cuda(), beta.cuda(),
                       x["scale"], h0=x["h0"].cuda(), cu_seqlens=x["cu_seqlens"].cuda())
    torch.cuda.synchronize()
    o, hT = o.cpu().float(), hT.cpu()
    cu = x["cu_seqlens"]
    for n in (0, 37, 63):
        a, b = int(cu[n]), int(cu[n + 1])
        sl = lambda t: t[a:b].contiguous()
        o_ref, h_ref = oracle.gdn_recurrent(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(beta),
                                            x["scale"], h0=x["h0"][n:n + 1],
                                            cu_seqlens=torch.tensor([0, b - a], dtype=torch.int64))
        assert oracle.rel_fro(o[a:b], o_ref) <= O_TOL
        assert oracle.rel_fro(hT[n:n + 1], h_ref) <= S_TOL


def test_gdn_prefill_no_tokens(sg):
    # packed call whose sequences are all empty: no output rows, hT = h0 (zeros without h0)
    H = 3
    q = torch.empty((0, H, 128), dtype=torch.bfloat16, device="cuda")
    g = torch.empty((0, H), dtype=torch.float32, device="cuda")
    cu = torch.zeros(4, dtype=torch.int64, device="cuda")
    h0 = inputs.make_decode_state("gdn_decode", nseq=3, H=H)
    o, hT = sg.gdn_fwd(q, q.clone(), q.clone(), g, g.clone(), 0.088, h0=h0.cuda(), cu_seqlens=cu)
    _, hz = sg.gdn_fwd(q, q.clone(), q.clone(), g, g.clone(), 0.088, cu_seqlens=cu)
    torch.cuda.synchronize()
    assert o.numel() == 0
    assert torch.equal(hT.cpu(), h0)
    assert torch.count_nonzero(hz).item() == 0

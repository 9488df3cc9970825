"""Parity of the chunked gated delta rule (sala_gla_gdn_chunk_fwd, through the C ABI) with the
fp64 oracle's recurrence (oracle.gdn_recurrent, "Formulas and Code for Adapting Inference to
GDN/KDA Linear Modules", section 1.1; the chunked form of section 1.2 computes the same).

Tolerances as for the Simple GLA prefill: relative Frobenius error <= 1e-2 for o and <= 5e-3
for the final states, over whole tensors and per (sequence, head) (sequences shorter than one
chunk pooled per head, as in test_gpu_parity).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_attention_gb300 import inputs
from parity_report import record

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
S_TOL = 5e-3
CHUNK = 64


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_linear_attention_gb300 import build, sala_gla
    build.build()
    return sala_gla


def _inputs(lens, H, seed):
    x = inputs.make_prefill("varlen", seqlens=tuple(lens), H=H, seed=seed)
    gen = torch.Generator().manual_seed(seed)
    beta = torch.sigmoid(torch.randn(x["g"].shape, generator=gen))
    return x, beta


def _run(sg, x, beta, g=None):
    g = x["g"] if g is None else g
    o, hT = sg.gdn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), g.cuda(), beta.cuda(),
                       x["scale"], h0=None if x["h0"] is None else x["h0"].cuda(),
                       cu_seqlens=None if x["cu_seqlens"] is None else x["cu_seqlens"].cuda(),
                       chunked=True)
    torch.cuda.synchronize()
    assert sg.get_device_status() == 0
    return o.cpu().float(), hT.cpu()


def _check(o, hT, o_ref, h_ref, bounds):
    of = o.reshape(o_ref.shape)
    assert oracle.rel_fro(of, o_ref) <= O_TOL
    assert oracle.rel_fro(hT, h_ref) <= S_TOL
    res = {}
    long_b = [(a, b) for a, b in bounds if b - a >= CHUNK]
    short_rows = [r for a, b in bounds if 0 < b - a < CHUNK for r in range(a, b)]
    if long_b:
        so = oracle.rel_fro_slices(of, o_ref, long_b)
        assert so.max() <= O_TOL, f"worst (sequence, head) output error {so.max():.3e}"
        res["o_slice_max"] = float(so.max())
    if short_rows:
        ss = oracle.rel_fro_slices(of[short_rows], o_ref[short_rows], [(0, len(short_rows))])
        assert ss.max() <= O_TOL
        res["o_short_block_max"] = float(ss.max())
    sh = oracle.rel_fro_slices(hT, h_ref, [(n, n + 1) for n in range(hT.shape[0])])
    assert sh.max() <= S_TOL, f"worst (sequence, head) state error {sh.max():.3e}"
    res["hT_slice_max"] = float(sh.max())
    record(res)


@pytest.mark.parametrize("lens", [[1], [63], [64], [65], [200], [1000], [5, 0, 130, 64],
                                  [700, 300], [64] * 5])
def test_gdn_chunk_packed(sg, lens):
    x, beta = _inputs(lens, 3, seed=sum(lens) + len(lens))
    o, hT = _run(sg, x, beta)
    o_ref, h_ref = oracle.gdn_recurrent(x["q"], x["k"], x["v"], x["g"], beta, x["scale"],
                                        h0=x["h0"], cu_seqlens=x["cu_seqlens"])
    _check(o, hT, o_ref, h_ref, oracle.seq_bounds(x["cu_seqlens"]))
    for n, L in enumerate(lens):                 # an empty sequence returns h0
        if L == 0:
            assert torch.equal(hT[n], x["h0"][n])


def test_gdn_chunk_rows_without_state(sg):
    # B = 3 rows of 96 tokens, no h0
    x, beta = _inputs([96] * 3, 2, seed=21)
    q, k, v = (x[n].reshape(3, 96, 2, 128) for n in ("q", "k", "v"))
    g, b = x["g"].reshape(3, 96, 2), beta.reshape(3, 96, 2)
    xr = dict(q=q, k=k, v=v, g=g, h0=None, cu_seqlens=None, scale=x["scale"])
    o, hT = _run(sg, xr, b)
    o_ref, h_ref = oracle.gdn_recurrent(q, k, v, g, b, x["scale"])
    _check(o, hT, o_ref, h_ref, [(96 * i, 96 * (i + 1)) for i in range(3)])


def test_gdn_chunk_strong_and_zero_gates(sg):
    # gates of 0 (no decay), single very strong gates and a run of strong decay: every factor
    # of the chunked form stays within [0, 1]
    x, beta = _inputs([300, 90], 2, seed=43)
    g = x["g"].clone()
    g[:40] = 0.0
    g[50, 0] = -60.0
    g[100:140] = -3.0
    g[230] = -200.0
    o, hT = _run(sg, x, beta, g=g)
    o_ref, h_ref = oracle.gdn_recurrent(x["q"], x["k"], x["v"], g, beta, x["scale"],
                                        h0=x["h0"], cu_seqlens=x["cu_seqlens"])
    assert torch.isfinite(o).all() and torch.isfinite(hT).all()
    _check(o, hT, o_ref, h_ref, oracle.seq_bounds(x["cu_seqlens"]))


def test_gdn_chunk_beta_zero_is_decay_only(sg):
    # beta = 0: no writes, the state only decays and the output reads it
    x, _ = _inputs([150], 2, seed=45)
    beta = torch.zeros_like(x["g"])
    o, hT = _run(sg, x, beta)
    o_ref, h_ref = oracle.gdn_recurrent(x["q"], x["k"], x["v"], x["g"], beta, x["scale"],
                                        h0=x["h0"], cu_seqlens=x["cu_seqlens"])
    _check(o, hT, o_ref, h_ref, oracle.seq_bounds(x["cu_seqlens"]))


def test_gdn_chunk_bench_size_sampled(sg):
    # the benchmark's workload and launch (64 sequences x 256 tokens, 32 heads); three
    # sequences checked against the oracle, every one against the recurrent kernel
    lens = (256,) * 64
    x = inputs.make_prefill("varlen", seqlens=lens, H=32, seed=13)
    beta = torch.sigmoid(torch.randn(x["g"].shape, generator=torch.Generator().manual_seed(13)))
    o, hT = _run(sg, x, beta)
    o_rec, h_rec = sg.gdn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), x["g"].cuda(),
                              beta.cuda(), x["scale"], h0=x["h0"].cuda(),
                              cu_seqlens=x["cu_seqlens"].cuda())
    torch.cuda.synchronize()
    assert oracle.rel_fro(o, o_rec.cpu().float()) <= O_TOL
    assert oracle.rel_fro(hT, h_rec.cpu()) <= S_TOL
    cu = x["cu_seqlens"]
    for n in (0, 37, 63):
        a, b = int(cu[n]), int(cu[n + 1])
        sl = lambda t: t[a:b].contiguous()
        o_ref, h_ref = oracle.gdn_recurrent(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), sl(beta),
                                            x["scale"], h0=x["h0"][n:n + 1],
                                            cu_seqlens=torch.tensor([0, b - a], dtype=torch.int64))
        _check(o[a:b], hT[n:n + 1], o_ref, h_ref, [(0, b - a)])


def test_gdn_chunk_one_long_sequence(sg):
    # one sequence of 16,384 tokens, 32 heads (the new_v pass runs 32 CTAs, the prefill that
    # follows is segment-parallel); four heads checked against the oracle
    x = inputs.make_prefill("varlen", seqlens=(16384,), H=32, seed=47)
    beta = torch.sigmoid(torch.randn(x["g"].shape, generator=torch.Generator().manual_seed(47)))
    o, hT = _run(sg, x, beta)
    heads = [0, 9, 22, 31]
    sel = lambda t: t[:, heads].contiguous()
    o_ref, h_ref = oracle.gdn_recurrent(sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["g"]),
                                        sel(beta), x["scale"], h0=x["h0"][:, heads],
                                        cu_seqlens=x["cu_seqlens"])
    _check(o[:, heads], hT[:, heads], o_ref, h_ref, [(0, 16384)])

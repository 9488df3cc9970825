"""Seeded randomized parity: many small varlen configurations drawn from a fixed generator,
each checked against the fp64 oracle over whole tensors and every (sequence, head) slice
(sequences shorter than one chunk pooled per head, as in test_gpu_parity).

The lengths mix empty and 1-token sequences, chunk boundaries (63, 64, 65, 127, 128, 129) and
sequences long enough for several segments; head counts vary; some configurations scale one
head's log-decays so that chunks take the exact route and the reference point moves. Covered:
the Simple GLA prefill (sala_gla_chunk_fwd), the chunked gated delta rule
(sala_gla_gdn_chunk_fwd) and the q/k prologue (sala_gla_qk_prologue).
"""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_attention_gb300 import inputs

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
S_TOL = 5e-3
CHUNK = 64
LENGTHS = [0, 1, 2, 17, 63, 64, 65, 127, 128, 129, 200, 639, 640, 641, 700, 1001, 1300, 1500]
N_CASES = 12


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_linear_attention_gb300 import build, sala_gla
    build.build()
    return sala_gla


def _case(i):
    rng = np.random.default_rng([20261202, i])
    nseq = int(rng.integers(1, 9))
    lens = [int(x) for x in rng.choice(LENGTHS, size=nseq)]
    if sum(lens) == 0:
        lens[0] = 65
    H = int(rng.choice([1, 2, 3, 5, 8]))
    strong = bool(rng.integers(0, 2))
    return lens, H, strong


def _slice_check(o, hT, o_ref, h_ref, cu):
    of = o.reshape(o_ref.shape)
    assert oracle.rel_fro(of, o_ref) <= O_TOL
    assert oracle.rel_fro(hT, h_ref) <= S_TOL
    bounds = oracle.seq_bounds(cu)
    long_b = [(a, b) for a, b in bounds if b - a >= CHUNK]
    short_rows = [r for a, b in bounds if 0 < b - a < CHUNK for r in range(a, b)]
    if long_b:
        assert oracle.rel_fro_slices(of, o_ref, long_b).max() <= O_TOL
    if short_rows:
        assert oracle.rel_fro_slices(of[short_rows], o_ref[short_rows], [(0, len(short_rows))]).max() <= O_TOL
    sh = oracle.rel_fro_slices(hT, h_ref, [(n, n + 1) for n in range(hT.shape[0])])
    assert sh.max() <= S_TOL


def _inputs(i):
    lens, H, strong = _case(i)
    x = inputs.make_prefill("varlen", seqlens=tuple(lens), H=H, seed=1000 + i)
    g = x["g"].clone()
    if strong:
        g[:, 0] = g[:, 0] * 60.0   # head 0: chunks with wide decay ranges (exact route)
    return x, g, lens, H


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_prefill(sg, i):
    x, g, lens, H = _inputs(i)
    o, hT = sg.chunk_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), g.cuda(), x["scale"],
                         h0=x["h0"].cuda(), cu_seqlens=x["cu_seqlens"].cuda())
    torch.cuda.synchronize()
    assert sg.get_device_status() == 0
    o_ref, h_ref = oracle.recurrent(x["q"], x["k"], x["v"], g, x["scale"], h0=x["h0"],
                                    cu_seqlens=x["cu_seqlens"])
    _slice_check(o.cpu().float(), hT.cpu(), o_ref, h_ref, x["cu_seqlens"])


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_gdn_chunked(sg, i):
    x, g, lens, H = _inputs(i)
    gen = torch.Generator().manual_seed(2000 + i)
    beta = torch.sigmoid(torch.randn(g.shape, generator=gen))
    o, hT = sg.gdn_fwd(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(), g.cuda(), beta.cuda(),
                       x["scale"], h0=x["h0"].cuda(), cu_seqlens=x["cu_seqlens"].cuda(), chunked=True)
    torch.cuda.synchronize()
    assert sg.get_device_status() == 0
    o_ref, h_ref = oracle.gdn_recurrent(x["q"], x["k"], x["v"], g, beta, x["scale"], h0=x["h0"],
                                        cu_seqlens=x["cu_seqlens"])
    _slice_check(o.cpu().float(), hT.cpu(), o_ref, h_ref, x["cu_seqlens"])


@pytest.mark.parametrize("i", range(N_CASES))
def test_fuzz_prologue(sg, i):
    lens, H, _ = _case(i)
    T = sum(lens)
    gen = torch.Generator().manual_seed(3000 + i)
    q = (3 * torch.randn((T, H, 128), generator=gen)).to(torch.bfloat16)
    k = (3 * torch.randn((T, H, 128), generator=gen)).to(torch.bfloat16)
    qw = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    start = torch.randint(0, 50000, (len(lens),), generator=gen, dtype=torch.int64)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    qd, kd = q.cuda(), k.cuda()
    sg.qk_prologue(qd, kd, qw.cuda(), kw.cuda(), 1e-6, 10000.0, cu_seqlens=cu.cuda(),
                   start_pos=start.cuda())
    torch.cuda.synchronize()
    assert sg.get_device_status() == 0
    pos = np.concatenate([np.arange(L) + int(start[n]) for n, L in enumerate(lens)])
    assert oracle.rel_fro(qd.cpu().float(), oracle.qk_prologue(q, qw, pos[:, None])) <= 5e-3
    k_ref = oracle.qk_prologue(k, kw, pos[:, None])
    assert oracle.rel_fro(kd.cpu().float(), k_ref) <= 5e-3
    # every token and head on its own (the prologue is per (token, head))
    err = oracle.rel_fro_slices(kd.cpu().float(), k_ref, [(t, t + 1) for t in range(T)])
    assert err.max() <= 2e-2

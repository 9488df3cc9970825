"""Parity of the q/k prologue (per-head RMSNorm with a weight, RoPE theta = 10000) with the
oracle: on its own in place on a prefill's q and k (sala_gla_qk_prologue), and fused into the
pooled decode step (sala_gla_recurrent_step_indexed with a prologue)."""
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


def _weights(seed):
    gen = torch.Generator().manual_seed(seed)
    qw = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    kw = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    return qw, kw


def _raw_tokens(T, H, seed):
    gen = torch.Generator().manual_seed(seed)
    return (3 * torch.randn((T, H, 128), generator=gen)).to(torch.bfloat16), \
           (3 * torch.randn((T, H, 128), generator=gen)).to(torch.bfloat16)


@pytest.mark.parametrize("lens,start", [([1], None), ([300], None), ([5, 0, 130, 64], [0, 7, 1000, 123456]),
                                        ([2048] * 2, [0, 4096])])
def test_prologue_prefill_packed(sg, lens, start):
    T, H = sum(lens), 4
    q, k = _raw_tokens(T, H, seed=T)
    qw, kw = _weights(1)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    sp = torch.tensor(start, dtype=torch.int64) if start is not None else None
    qd, kd = q.cuda(), k.cuda()
    sg.qk_prologue(qd, kd, qw.cuda(), kw.cuda(), 1e-6, 10000.0, cu_seqlens=cu.cuda(),
                   start_pos=sp.cuda() if sp is not None else None)
    torch.cuda.synchronize()
    pos = np.concatenate([np.arange(L) + (start[n] if start else 0) for n, L in enumerate(lens)])
    q_ref = oracle.qk_prologue(q, qw, pos[:, None])
    k_ref = oracle.qk_prologue(k, kw, pos[:, None])
    # both sides round to bf16; they may differ by one bf16 step where fp32 and fp64 round
    # differently
    assert oracle.rel_fro(qd.cpu().float(), q_ref) <= 5e-3
    assert oracle.rel_fro(kd.cpu().float(), k_ref) <= 5e-3
    assert np.mean(qd.cpu().double().numpy() == q_ref) > 0.95


@pytest.mark.parametrize("H", [32, 40])
def test_prologue_prefill_wide(sg, H):
    # 32 heads: four per warp in one group; 40: a second group per warp, partly past H
    lens = [37, 200]
    T = sum(lens)
    q, k = _raw_tokens(T, H, seed=H)
    qw, kw = _weights(3)
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    qd, kd = q.cuda(), k.cuda()
    sg.qk_prologue(qd, kd, qw.cuda(), kw.cuda(), 1e-6, 10000.0, cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    pos = np.concatenate([np.arange(L) for L in lens])
    q_ref = oracle.qk_prologue(q, qw, pos[:, None])
    k_ref = oracle.qk_prologue(k, kw, pos[:, None])
    assert oracle.rel_fro(qd.cpu().float(), q_ref) <= 5e-3
    assert oracle.rel_fro(kd.cpu().float(), k_ref) <= 5e-3
    assert np.mean(kd.cpu().double().numpy() == k_ref) > 0.95
    # every head of every token, separately
    err = oracle.rel_fro_slices(kd.cpu().float(), k_ref, [(t, t + 1) for t in range(T)])
    assert err.max() <= 2e-2, f"worst (token, head) error {err.max():.3e}"


def test_prologue_prefill_rows(sg):
    # B = 2 rows of 100 tokens without cu_seqlens: positions restart per row
    q, k = _raw_tokens(200, 3, seed=5)
    qw, kw = _weights(2)
    qd, kd = q.reshape(2, 100, 3, 128).cuda(), k.reshape(2, 100, 3, 128).cuda()
    sg.qk_prologue(qd, kd, qw.cuda(), kw.cuda())
    torch.cuda.synchronize()
    pos = np.concatenate([np.arange(100), np.arange(100)])
    assert oracle.rel_fro(qd.cpu().reshape(200, 3, 128).float(), oracle.qk_prologue(q, qw, pos[:, None])) <= 5e-3


def test_dependent_launches_read_what_the_previous_one_wrote(sg):
    # the prologue and the output gate go out as programmatic dependents of the kernel before
    # them: back-to-back calls on the same tensors (each reading the previous one's output),
    # with no synchronisation in between, must give the oracle applied in sequence
    T, H = 4096, 8
    q, k = _raw_tokens(T, H, seed=21)
    qw, kw = _weights(4)
    qd, kd = q.cuda(), k.cuda()
    cu = torch.tensor([0, T], dtype=torch.int64)
    for _ in range(3):
        sg.qk_prologue(qd, kd, qw.cuda(), kw.cuda(), 1e-6, 10000.0, cu_seqlens=cu.cuda())
    gen = torch.Generator().manual_seed(22)
    z = torch.randn((T, H * 128), generator=gen).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(H * 128, generator=gen)).to(torch.bfloat16)
    out = torch.empty((T, H * 128), dtype=torch.bfloat16, device="cuda")
    sg.output_norm_gate(qd.reshape(T, H * 128), z.cuda(), w.cuda(), 1e-6, out=out)
    torch.cuda.synchronize()
    pos = np.arange(T)[:, None]
    q_ref, k_ref = q, k
    for _ in range(3):
        q_ref = torch.from_numpy(oracle.qk_prologue(q_ref, qw, pos)).to(torch.bfloat16)
        k_ref = torch.from_numpy(oracle.qk_prologue(k_ref, kw, pos)).to(torch.bfloat16)
    assert oracle.rel_fro(qd.cpu().float(), q_ref.float()) <= 1e-2
    assert oracle.rel_fro(kd.cpu().float(), k_ref.float()) <= 1e-2
    g_ref = oracle.output_norm_gate(qd.cpu().reshape(T, H * 128), z, w)
    assert oracle.rel_fro(out.cpu().float(), g_ref) <= 1e-2


def test_prologue_then_prefill_matches_oracle(sg):
    # the layer's path: prologue in place, then the chunked prefill
    x = inputs.make_prefill("varlen", seqlens=(700, 300), H=4, seed=17)
    qw, kw = _weights(3)
    q, k = x["q"].clone(), x["k"].clone()
    qd, kd = q.cuda(), k.cuda()
    cu = x["cu_seqlens"]
    sg.qk_prologue(qd, kd, qw.cuda(), kw.cuda(), cu_seqlens=cu.cuda())
    o, hT = sg.chunk_fwd(qd, kd, x["v"].cuda(), x["g"].cuda(), x["scale"], h0=x["h0"].cuda(),
                         cu_seqlens=cu.cuda())
    torch.cuda.synchronize()
    pos = np.concatenate([np.arange(700), np.arange(300)])
    qp = torch.from_numpy(oracle.qk_prologue(q, qw, pos[:, None])).to(torch.bfloat16)
    kp = torch.from_numpy(oracle.qk_prologue(k, kw, pos[:, None])).to(torch.bfloat16)
    o_ref, h_ref = oracle.recurrent(qp, kp, x["v"], x["g"], x["scale"], h0=x["h0"], cu_seqlens=cu)
    assert oracle.rel_fro(o.cpu().float(), o_ref) <= O_TOL
    assert oracle.rel_fro(hT.cpu(), h_ref) <= S_TOL


@pytest.mark.parametrize("storage", ["f32", "bf16"])
def test_prologue_fused_in_pooled_decode(sg, storage):
    N, H, P, steps = 6, 3, 9, 4
    qw, kw = _weights(4)
    p = inputs.make_decode_pool(nseq=N, H=H, pool=P, storage=storage, pad=(2,))
    x = inputs.make_decode_steps("decode_pool", 0, steps, nseq=N, H=H)
    gen = torch.Generator().manual_seed(9)
    # raw (unnormalised) projections
    qr = (3 * torch.randn((steps, N, H, 128), generator=gen)).to(torch.bfloat16)
    kr = (3 * torch.randn((steps, N, H, 128), generator=gen)).to(torch.bfloat16)
    pos0 = torch.tensor([5, 900, 0, 17, 31000, 64], dtype=torch.int64)
    pool = p["pool"].cuda().clone()
    idx = p["indices"].cuda()
    ref = p["pool"]
    for s in range(steps):
        pos = pos0 + s
        o = sg.recurrent_step_indexed(qr[s].cuda(), kr[s].cuda(), x["v"][s].cuda(), x["g"][s].cuda(),
                                      x["scale"], pool, idx, prologue=(qw.cuda(), kw.cuda(), 1e-6, 10000.0),
                                      positions=pos.cuda())
        torch.cuda.synchronize()
        qp = torch.from_numpy(oracle.qk_prologue(qr[s], qw, pos.numpy()[:, None])).to(torch.bfloat16)
        kp = torch.from_numpy(oracle.qk_prologue(kr[s], kw, pos.numpy()[:, None])).to(torch.bfloat16)
        o_ref, ref = oracle.recurrent_step_indexed(qp, kp, x["v"][s], x["g"][s], x["scale"], ref,
                                                   p["indices"], storage=storage)
        if storage == "bf16":
            ref = torch.from_numpy(ref).to(torch.bfloat16)
        assert oracle.rel_fro(o.cpu().float(), o_ref) <= O_TOL
        assert torch.all(o[2].cpu() == 0)
    named = [int(i) for i in p["indices"] if i >= 0]
    assert oracle.rel_fro(pool.cpu()[named].float(), oracle._as_f64(ref)[named]) <= S_TOL
    # q and k themselves are not modified by the fused prologue

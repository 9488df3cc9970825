"""Seeded synthetic inputs for the Simple GLA prefill and decode workloads.

This module is shared by the tests, the benchmark and the oracle checks, and holds none of
the recurrence's arithmetic: it only draws random numbers and applies the input
preparation that the workloads prescribe before the kernel sees its operands (q/k
normalisation, the log-sigmoid gate, the fixed per-head decay), all in float32 before the
cast to bfloat16 (round to nearest even).

Random stream. Every tensor is drawn in token blocks; block ``b`` of stream ``s`` under
seed ``seed`` comes from ``numpy.random.default_rng([seed, s, b])``. Blocks are independent,
so they are drawn on a thread pool and any block can be regenerated alone; the values do
not depend on the number of threads.

Shapes of the pages' model (MiniCPM-SALA lightning layers): 32 heads of dimension 128.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

D = 128
BLOCK_TOKENS = 1024

# stream ids
_Q, _K, _V, _U, _H0, _SLOT, _Z, _W, _QW, _KW, _BETA = 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                   # "prefill" or "decode"
    H: int
    seqlens: tuple              # prefill: one entry per sequence; decode: () (see nseq)
    qk_norm: str                # "l2" or "rms"
    gate: str                   # "logsigmoid" or "const"
    h0: bool                    # nonzero initial state
    seed: int
    varlen: bool = False
    nseq: int = 0               # decode: number of sequences
    steps: int = 0              # decode: consecutive steps
    pool: int = 0               # pooled decode: slots in the state pool
    storage: str = "f32"        # pooled decode: state storage type ("f32" or "bf16")
    description: str = field(default="", compare=False)

    @property
    def T(self) -> int:
        return int(sum(self.seqlens))


WORKLOADS = {
    "tiny": Workload(
        "tiny", "prefill", H=4, seqlens=(256,), qk_norm="l2", gate="logsigmoid", h0=False,
        seed=0, description="tiny prefill: B=1, H=4, T=256; q,k L2-normalised; "
        "g=logsigmoid(u), u~U(2,6); h0=0"),
    "sala_layer": Workload(
        "sala_layer", "prefill", H=32, seqlens=(8192,), qk_norm="rms", gate="const", h0=False,
        seed=1, description="MiniCPM-SALA lightning-layer prefill: B=1, H=32, T=8192; q,k "
        "RMS-normalised; g_h=-2^(-8(h+1)/32) for every token; h0=0"),
    "varlen": Workload(
        "varlen", "prefill", H=32, seqlens=(512, 1024, 2048, 4096, 8192, 16384, 16384, 17920),
        qk_norm="l2", gate="logsigmoid", h0=True, seed=2, varlen=True,
        description="varlen packed prefill: 8 sequences, 65536 tokens; q,k L2-normalised; "
        "g=logsigmoid(u), u~U(2,6); h0~N(0,0.02)"),
    "long": Workload(
        "long", "prefill", H=32, seqlens=(131072,), qk_norm="rms", gate="const", h0=True,
        seed=3, description="long-context prefill: B=1, H=32, T=131072; q,k RMS-normalised; "
        "g_h=-2^(-8(h+1)/32); h0~N(0,0.02)"),
    "decode": Workload(
        "decode", "decode", H=32, seqlens=(), qk_norm="l2", gate="logsigmoid", h0=True, seed=4,
        nseq=256, steps=1000, description="batched recurrent decode: 256 sequences x 1 token, "
        "H=32; q,k L2-normalised; g=logsigmoid(u), u~U(2,6); S~N(0,0.02) [256,32,128,128] "
        "fp32 updated in place; 1000 consecutive steps"),
    "gdn_decode": Workload(
        "gdn_decode", "decode", H=32, seqlens=(), qk_norm="l2", gate="logsigmoid", h0=True, seed=12,
        nseq=256, steps=1000, description="batched gated-delta-rule decode: 256 sequences x 1 "
        "token, H=32; q,k L2-normalised; g=logsigmoid(u), u~U(2,6); beta=sigmoid(w), w~N(0,1); "
        "S~N(0,0.02) [256,32,128,128] fp32 updated in place; 1000 consecutive steps"),
    "decode_pool": Workload(
        "decode_pool", "decode", H=32, seqlens=(), qk_norm="l2", gate="logsigmoid", h0=True,
        seed=4, nseq=256, steps=1000, pool=512, storage="bf16",
        description="pooled recurrent decode: 256 sequences x 1 token, H=32, states in a "
        "pool of 512 slots [512,32,128,128] stored in bf16 (256 MB read+written per step), "
        "slots of the batch = a seeded permutation of the pool; per-step q, k, v, g those of "
        "the decode workload (same seed); S~N(0,0.02); 1000 consecutive steps"),
}

SCALE = 1.0 / math.sqrt(D)     # 1/sqrt(128) = 0.08839...


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def _normal(seed: int, stream: int, block: int, shape) -> np.ndarray:
    return np.random.default_rng([seed, stream, block]).standard_normal(shape, dtype=np.float32)


def _uniform(seed: int, stream: int, block: int, shape, lo: float, hi: float) -> np.ndarray:
    r = np.random.default_rng([seed, stream, block]).random(shape, dtype=np.float32)
    return (lo + (hi - lo) * r).astype(np.float32)


def l2_normalise(x: torch.Tensor) -> torch.Tensor:
    """x * rsqrt(sum(x^2) + 1e-6) over the last dimension, in float32."""
    return x * torch.rsqrt((x * x).sum(-1, keepdim=True) + 1e-6)


def rms_normalise(x: torch.Tensor) -> torch.Tensor:
    """x / sqrt(mean(x^2) + 1e-6) over the last dimension (unit weight), in float32."""
    return x * torch.rsqrt((x * x).mean(-1, keepdim=True) + 1e-6)


def const_head_gate(H: int) -> torch.Tensor:
    """Fixed per-head log-decay g_h = -2^(-8(h+1)/H), h = 0..H-1 (float32)."""
    return torch.tensor([-(2.0 ** (-8.0 * (h + 1) / H)) for h in range(H)], dtype=torch.float32)


def _tokens(seed, stream, T, H, d, pool, post=None, dtype=torch.bfloat16):
    """Draw a [T, H, d] float32 normal tensor block by block, optionally post-process in
    float32, and cast."""
    out = torch.empty((T, H, d), dtype=dtype)
    nblk = (T + BLOCK_TOKENS - 1) // BLOCK_TOKENS

    def one(b):
        t0 = b * BLOCK_TOKENS
        n = min(BLOCK_TOKENS, T - t0)
        x = torch.from_numpy(_normal(seed, stream, b, (n, H, d)))
        if post is not None:
            x = post(x)
        out[t0:t0 + n] = x.to(dtype)

    list(pool.map(one, range(nblk)))
    return out


def _gate(w: Workload, T: int, pool) -> torch.Tensor:
    if w.gate == "const":
        return const_head_gate(w.H).expand(T, w.H).contiguous()
    g = torch.empty((T, w.H), dtype=torch.float32)
    nblk = (T + BLOCK_TOKENS - 1) // BLOCK_TOKENS

    def one(b):
        t0 = b * BLOCK_TOKENS
        n = min(BLOCK_TOKENS, T - t0)
        u = torch.from_numpy(_uniform(w.seed, _U, b, (n, w.H), 2.0, 6.0))
        g[t0:t0 + n] = torch.nn.functional.logsigmoid(u)

    list(pool.map(one, range(nblk)))
    return g


def _qk_post(w: Workload):
    return l2_normalise if w.qk_norm == "l2" else rms_normalise


def _states(seed: int, stream: int, n: int, H: int, pool) -> torch.Tensor:
    """[n, H, D, D] float32 ~ N(0, 0.02^2), one block per sequence."""
    out = torch.empty((n, H, D, D), dtype=torch.float32)

    def one(i):
        out[i] = torch.from_numpy(_normal(seed, stream, i, (H, D, D))) * 0.02

    list(pool.map(one, range(n)))
    return out


def make_prefill(w: Workload | str, *, seqlens=None, H=None, seed=None) -> dict:
    """Inputs of a prefill workload as CPU tensors.

    Returns a dict with q, k, v (bf16 [B, T, H, 128], or packed [T, H, 128] when the workload
    is varlen), g (fp32, same leading shape, last dim H), h0 (fp32 [nseq, H, 128, 128] or
    None), cu_seqlens (int64 [nseq+1] or None), scale, and the workload. ``seqlens``, ``H``
    and ``seed`` override the workload's sizes for small parity cases.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    assert w.kind == "prefill"
    if seqlens is not None or H is not None or seed is not None:
        sl = tuple(int(x) for x in (seqlens if seqlens is not None else w.seqlens))
        w = Workload(w.name, w.kind, H=H or w.H, seqlens=sl, qk_norm=w.qk_norm,
                     gate=w.gate, h0=w.h0, seed=w.seed if seed is None else seed,
                     varlen=w.varlen or len(sl) > 1, description=w.description)
    T, Hh = w.T, w.H
    with ThreadPoolExecutor(_threads()) as pool:
        post = _qk_post(w)
        q = _tokens(w.seed, _Q, T, Hh, D, pool, post)
        k = _tokens(w.seed, _K, T, Hh, D, pool, post)
        v = _tokens(w.seed, _V, T, Hh, D, pool)
        g = _gate(w, T, pool)
        nseq = len(w.seqlens)
        h0 = _states(w.seed, _H0, nseq, Hh, pool) if w.h0 else None
    if w.varlen:
        cu = torch.zeros(nseq + 1, dtype=torch.int64)
        cu[1:] = torch.cumsum(torch.tensor(w.seqlens, dtype=torch.int64), 0)
        return dict(q=q, k=k, v=v, g=g, h0=h0, cu_seqlens=cu, scale=SCALE, workload=w)
    return dict(q=q.unsqueeze(0), k=k.unsqueeze(0), v=v.unsqueeze(0), g=g.unsqueeze(0), h0=h0,
                cu_seqlens=None, scale=SCALE, workload=w)


def make_decode_state(w: Workload | str = "decode", *, nseq=None, H=None) -> torch.Tensor:
    """Initial decode states [nseq, H, 128, 128] fp32 ~ N(0, 0.02^2)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    with ThreadPoolExecutor(_threads()) as pool:
        return _states(w.seed, _H0, nseq or w.nseq, H or w.H, pool)


def make_decode_steps(w: Workload | str = "decode", start: int = 0, count: int | None = None,
                      *, nseq=None, H=None) -> dict:
    """Per-step decode inputs for steps [start, start+count).

    Returns q, k, v bf16 [count, nseq, H, 128] and g fp32 [count, nseq, H]. Step s draws
    block s of each stream, so any range of steps can be regenerated alone.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    count = w.steps - start if count is None else count
    n, Hh = nseq or w.nseq, H or w.H
    post = _qk_post(w)
    q = torch.empty((count, n, Hh, D), dtype=torch.bfloat16)
    k = torch.empty_like(q)
    v = torch.empty_like(q)
    g = torch.empty((count, n, Hh), dtype=torch.float32)

    def one(i):
        s = start + i
        q[i] = post(torch.from_numpy(_normal(w.seed, _Q, s, (n, Hh, D)))).to(torch.bfloat16)
        k[i] = post(torch.from_numpy(_normal(w.seed, _K, s, (n, Hh, D)))).to(torch.bfloat16)
        v[i] = torch.from_numpy(_normal(w.seed, _V, s, (n, Hh, D))).to(torch.bfloat16)
        u = torch.from_numpy(_uniform(w.seed, _U, s, (n, Hh), 2.0, 6.0))
        g[i] = torch.nn.functional.logsigmoid(u)

    with ThreadPoolExecutor(_threads()) as pool:
        list(pool.map(one, range(count)))
    return dict(q=q, k=k, v=v, g=g, scale=SCALE, workload=w)


def make_decode_pool(w: Workload | str = "decode_pool", *, nseq=None, H=None, pool=None,
                     storage=None, pad=()) -> dict:
    """Pool and slot indices of a pooled decode workload.

    Returns pool [P, H, 128, 128] (states ~ N(0, 0.02^2) drawn in float32; cast to bfloat16
    for bf16 storage) and indices int32 [nseq]: the first nseq entries of a seeded
    permutation of the P slots, with the rows listed in ``pad`` set to -1 (padding). The
    per-step q, k, v, g come from :func:`make_decode_steps` with the same workload.
    """
    if isinstance(w, str):
        w = WORKLOADS[w]
    n, Hh, P = nseq or w.nseq, H or w.H, pool or w.pool
    st = storage or w.storage
    assert n <= P
    with ThreadPoolExecutor(_threads()) as tp:
        S = _states(w.seed, _H0, P, Hh, tp)
    perm = np.random.default_rng([w.seed, _SLOT, 0]).permutation(P)[:n]
    idx = torch.from_numpy(perm.astype(np.int32))
    for r in pad:
        idx[r] = -1
    return dict(pool=S.to(torch.bfloat16) if st == "bf16" else S, indices=idx, storage=st,
                workload=w)


def make_output_gate(T: int = 8192, H: int = 32, seed: int = 6) -> dict:
    """Inputs of the output norm and gate: o ~ N(0, 1) and gate logits z ~ N(0, 2^2) as bf16
    [T, H, 128], norm weight w = 1 + 0.1 N(0, 1) as bf16 [H * 128]. The defaults are the
    lightning layer's prefill shape (8192 tokens, 32 heads)."""
    o = torch.empty((T, H, D), dtype=torch.bfloat16)
    z = torch.empty_like(o)
    nblk = (T + BLOCK_TOKENS - 1) // BLOCK_TOKENS

    def one(b):
        t0 = b * BLOCK_TOKENS
        n = min(BLOCK_TOKENS, T - t0)
        o[t0:t0 + n] = torch.from_numpy(_normal(seed, _Q, b, (n, H, D))).to(torch.bfloat16)
        z[t0:t0 + n] = (2.0 * torch.from_numpy(_normal(seed, _Z, b, (n, H, D)))).to(torch.bfloat16)

    with ThreadPoolExecutor(_threads()) as pool:
        list(pool.map(one, range(nblk)))
    w = (1.0 + 0.1 * torch.from_numpy(_normal(seed, _W, 0, (H * D,)))).to(torch.bfloat16)
    return dict(o=o, z=z, w=w, eps=1e-6)


def make_qk_prologue(T: int = 8192, H: int = 32, seed: int = 8) -> dict:
    """Raw (before the prologue) q, k ~ 3 N(0, 1) as bf16 [T, H, 128] and the RMSNorm weights
    q_weight, k_weight = 1 + 0.1 N(0, 1) as bf16 [128]; eps 1e-6, theta 10000. The defaults
    are the lightning layer's prefill shape."""
    q = torch.empty((T, H, D), dtype=torch.bfloat16)
    k = torch.empty_like(q)
    nblk = (T + BLOCK_TOKENS - 1) // BLOCK_TOKENS

    def one(b):
        t0 = b * BLOCK_TOKENS
        n = min(BLOCK_TOKENS, T - t0)
        q[t0:t0 + n] = (3.0 * torch.from_numpy(_normal(seed, _Q, b, (n, H, D)))).to(torch.bfloat16)
        k[t0:t0 + n] = (3.0 * torch.from_numpy(_normal(seed, _K, b, (n, H, D)))).to(torch.bfloat16)

    with ThreadPoolExecutor(_threads()) as pool:
        list(pool.map(one, range(nblk)))
    qw = (1.0 + 0.1 * torch.from_numpy(_normal(seed, _QW, 0, (D,)))).to(torch.bfloat16)
    kw = (1.0 + 0.1 * torch.from_numpy(_normal(seed, _KW, 0, (D,)))).to(torch.bfloat16)
    return dict(q=q, k=k, q_weight=qw, k_weight=kw, eps=1e-6, theta=10000.0)


def make_gdn_beta(w: Workload | str = "gdn_decode", start: int = 0, count: int | None = None,
                  *, nseq=None, H=None) -> torch.Tensor:
    """Write strengths of the gated delta rule for decode steps [start, start+count):
    beta = sigmoid(w), w ~ N(0, 1), fp32 [count, nseq, H] (stream 11, one block per step)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    count = w.steps - start if count is None else count
    n, Hh = nseq or w.nseq, H or w.H
    b = torch.empty((count, n, Hh), dtype=torch.float32)
    for i in range(count):
        b[i] = torch.sigmoid(torch.from_numpy(_normal(w.seed, _BETA, start + i, (n, Hh))))
    return b

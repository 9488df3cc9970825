"""fp64 CPU oracle for the Simple GLA hot path.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the library under ``gated_linear_attention_gb300``
never does, and this package imports nothing from it. The two share no code.

Three independent statements of the same computation:

* :func:`recurrent` -- the token-by-token recurrence in C (``recurrent.c``), fp64, on
  host threads. "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple
  GLA)", block "Simple GLA Recurrence": decay the state by exp(g), add k^T v, then
  read o = scale * q S.
* :func:`chunkwise` -- the chunked form with chunk size C, in numpy fp64, taking the steps
  of "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules", section 1.2
  (chunk decay from the cumulative sum of g, the masked decay matrix, the inter-chunk
  term (q * exp(g)) @ S, the intra-chunk term (q k^T * gamma).tril() @ v, and the state
  refresh S * exp(g_last) + (k * exp(g_last - g))^T @ v), specialised to the Simple GLA
  case: no delta rule, beta = 1, so the "new v" is v itself.
* :func:`bruteforce` -- the quadratic parallel form, written from the unrolled closed form
  of the same Blueprint page (section "Why Linear Attention Loses Information", Problem
  1: S_n = alpha^n S_0 + sum_i alpha^(n-i) k_i^T v_i) with a per-token decay:
  o_t = scale * [ sum_{j<=t} exp(G_t - G_j) (q_t . k_j) v_j + exp(G_t) q_t h0 ],
  G_t = sum_{i<=t} g_i within the sequence. For tiny inputs only.

Beside them, :func:`gdn_recurrent` and :func:`gdn_chunkwise` state the gated delta rule
(the second workload) in its two forms, :func:`qk_prologue` is the layer's per-head q/k
RMSNorm and RoPE,
:func:`output_norm_gate` is the layer's output RMSNorm and sigmoid gate, and
:func:`recurrent_step_indexed` is one decode step on states gathered from and
written back to a pool through slot indices (fp32 or bf16 storage), built on
:func:`recurrent`.

All of them take the exact values the GPU receives (bf16 q/k/v, fp32 g, fp32 h0) and compute
in float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_SRC = os.path.join(_HERE, "recurrent.c")
_lib = None
_lib_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``recurrent.c`` into ``oracle/_build/liboracle.so`` (plain gcc, -O2)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def load_library(path: str):
    """ctypes handle with the argument types of ``oracle_recurrent`` declared."""
    lib = ctypes.CDLL(path)
    p = ctypes.c_void_p
    i64 = ctypes.c_int64
    lib.oracle_recurrent.argtypes = [p, p, p, p, ctypes.c_double, p, p, i64, i64, i64,
                                     i64, p, i64, p, p, ctypes.c_int]
    lib.oracle_recurrent.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            build()
            _lib = load_library(_LIB_PATH)
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ----------------------------------------------------------------------------------------
# argument helpers (no arithmetic of the method here)


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    assert x.dtype == torch.bfloat16 and x.device.type == "cpu"
    return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))


def _as_f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu()
        if x.dtype == torch.bfloat16:
            x = x.float()
        x = x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _packed(q, k, v, g, cu_seqlens):
    """Flatten [B, T, H, d] to the packed [B*T, H, d] form and build cu_seqlens."""
    if q.dim() == 4:
        B, T = q.shape[0], q.shape[1]
        q, k, v = (x.reshape(B * T, *x.shape[2:]) for x in (q, k, v))
        g = g.reshape(B * T, g.shape[-1])
        if cu_seqlens is None:
            cu_seqlens = torch.arange(0, B + 1, dtype=torch.int64) * T
    elif cu_seqlens is None:
        cu_seqlens = torch.tensor([0, q.shape[0]], dtype=torch.int64)
    cu = np.ascontiguousarray(torch.as_tensor(cu_seqlens).cpu().numpy().astype(np.int64))
    return q, k, v, g, cu


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


# ----------------------------------------------------------------------------------------
# the recurrence (C, fp64)


def recurrent(q, k, v, g, scale, h0=None, cu_seqlens=None, heads=None, want_o=True,
              nthreads: int | None = None, _lib=None):
    """Token-by-token fp64 recurrence.

    q, k: bf16 [B, T, H, dk] or packed [T, H, dk]; v: bf16 [..., dv]; g: fp32 [B, T, H] or
    [T, H]; h0: fp32/fp64 [nseq, H, dk, dv] or None; cu_seqlens: int64 [nseq+1] for packed
    input. ``heads`` selects a subset of heads (outputs then hold only those heads, in that
    order). Returns (o [T_total, nh, dv] float64 or None, hT [nseq, nh, dk, dv] float64).
    ``_lib`` substitutes another build of ``recurrent.c`` (the mutation tests use it).
    """
    lib = _lib or _load()
    q, k, v, g, cu = _packed(q, k, v, g, cu_seqlens)
    T, H, dk = q.shape
    dv = v.shape[-1]
    nseq = len(cu) - 1
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    gf = np.ascontiguousarray(g.float().numpy() if isinstance(g, torch.Tensor) else
                              np.asarray(g, dtype=np.float32))
    h0d = None if h0 is None else _as_f64(h0).reshape(nseq, H, dk, dv)
    hs = None if heads is None else np.ascontiguousarray(np.asarray(heads, dtype=np.int64))
    nh = H if hs is None else len(hs)
    o = np.empty((T, nh, dv), dtype=np.float64) if want_o else None
    hT = np.empty((nseq, nh, dk, dv), dtype=np.float64)
    rc = lib.oracle_recurrent(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gf), float(scale), _ptr(h0d),
                              _ptr(cu), nseq, H, dk, dv, _ptr(hs), nh, _ptr(o), _ptr(hT),
                              int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle_recurrent rejected its arguments (code {rc})")
    return o, hT


# ----------------------------------------------------------------------------------------
# the chunked form (numpy, fp64)


def _chunkwise_one(q, k, v, g, scale, S, C):
    """One sequence, one head: q, k [L, dk], v [L, dv], g [L], S [dk, dv] (all fp64)."""
    L = q.shape[0]
    o = np.empty((L, v.shape[1]), dtype=np.float64)
    for c0 in range(0, L, C):
        qi, ki, vi, gi = q[c0:c0 + C], k[c0:c0 + C], v[c0:c0 + C], g[c0:c0 + C]
        b = np.cumsum(gi)                               # chunk decay: cumulative sum of g
        gamma = np.exp(np.tril(b[:, None] - b[None, :]))  # masked difference, then exp
        o_inter = (qi * np.exp(b)[:, None]) @ S
        o_intra = np.tril(qi @ ki.T * gamma) @ vi
        o[c0:c0 + C] = scale * (o_inter + o_intra)
        S = S * np.exp(b[-1]) + (ki * np.exp(b[-1] - b)[:, None]).T @ vi   # state refresh
    return o, S


def chunkwise(q, k, v, g, scale, h0=None, cu_seqlens=None, chunk: int = 64):
    """Chunked fp64 form. Same arguments and return shapes as :func:`recurrent` (all heads)."""
    q, k, v, g, cu = _packed(q, k, v, g, cu_seqlens)
    qd, kd, vd, gd = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(g)
    T, H, dk = qd.shape
    dv = vd.shape[-1]
    nseq = len(cu) - 1
    h0d = None if h0 is None else _as_f64(h0).reshape(nseq, H, dk, dv)
    o = np.zeros((T, H, dv), dtype=np.float64)
    hT = np.zeros((nseq, H, dk, dv), dtype=np.float64)
    for n in range(nseq):
        s, e = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S0 = np.zeros((dk, dv)) if h0d is None else h0d[n, h].copy()
            o[s:e, h], hT[n, h] = _chunkwise_one(qd[s:e, h], kd[s:e, h], vd[s:e, h],
                                                 gd[s:e, h], scale, S0, chunk)
    return o, hT


# ----------------------------------------------------------------------------------------
# the quadratic parallel form (numpy, fp64, tiny inputs)


def bruteforce(q, k, v, g, scale, h0=None, cu_seqlens=None):
    """Quadratic fp64 form. Same arguments and return shapes as :func:`chunkwise`."""
    q, k, v, g, cu = _packed(q, k, v, g, cu_seqlens)
    qd, kd, vd, gd = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(g)
    T, H, dk = qd.shape
    dv = vd.shape[-1]
    nseq = len(cu) - 1
    h0d = None if h0 is None else _as_f64(h0).reshape(nseq, H, dk, dv)
    o = np.zeros((T, H, dv), dtype=np.float64)
    hT = np.zeros((nseq, H, dk, dv), dtype=np.float64)
    for n in range(nseq):
        s, e = int(cu[n]), int(cu[n + 1])
        L = e - s
        for h in range(H):
            G = np.cumsum(gd[s:e, h])
            # weight of token j in the state seen by token t: exp(G_t - G_j) for j <= t
            W = np.zeros((L, L))
            for t in range(L):
                W[t, :t + 1] = np.exp(G[t] - G[:t + 1])
            qk = qd[s:e, h] @ kd[s:e, h].T
            o_n = (W * qk) @ vd[s:e, h]
            S0 = np.zeros((dk, dv)) if h0d is None else h0d[n, h]
            if L:
                o_n += np.exp(G)[:, None] * (qd[s:e, h] @ S0)
            o[s:e, h] = scale * o_n
            # final state: exp(G_L - G_j) k_j^T v_j summed, plus exp(G_L) h0
            GL = G[-1] if L else 0.0
            w_end = np.exp(GL - G) if L else np.zeros(0)
            hT[n, h] = np.exp(GL) * S0 + (kd[s:e, h] * w_end[:, None]).T @ vd[s:e, h]
    return o, hT


# ----------------------------------------------------------------------------------------
# one decode step on states held in a pool (fp64)


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even), returned as
    float64. bfloat16 keeps 8 significant bits (the leading one included) and float32's
    exponent range; valid for values in the normal range of bfloat16 and for zero."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                    # x = m 2^e with 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)   # numpy rounds halves to even


def recurrent_step_indexed(q, k, v, g, scale, pool, indices, storage: str = "f32"):
    """One decode step on states kept in a pool and addressed by slot, in float64.

    "MiniCPM-SALA — Complete Blueprint", section "Memory Architecture": every request keeps
    its temporal state in a slot of a per-layer pool (1 MB per request in bf16 for 32
    heads); the decode step loads the state from its slot, applies the recurrence of
    section "B2 lightning-attn (Simple GLA)" (decay, k^T v update, o = scale q S) and saves
    the updated state back to the same slot. Row n uses slot indices[n]; a negative slot is
    a padding row (o = 0, no state read or written). With ``storage="bf16"`` the pool holds
    bfloat16 values: they are widened exactly, o reads the updated state before rounding,
    and the stored state is the updated state rounded to the nearest bfloat16.

    q, k, v: bf16 [N, H, dk|dv]; g: fp32 [N, H]; pool: [P, H, dk, dv] (float32/float64, or
    bfloat16 for "bf16"); indices: ints [N]. Returns (o [N, H, dv] float64, new pool
    [P, H, dk, dv] float64 holding the stored values). The recurrence itself is
    :func:`recurrent`, run on one-token sequences.
    """
    idx = np.asarray(indices.cpu() if isinstance(indices, torch.Tensor) else indices,
                     dtype=np.int64)
    P = pool.shape[0]
    if np.any(idx >= P):
        raise ValueError("slot index at or past the pool size")
    live = np.nonzero(idx >= 0)[0]
    if len(set(idx[live].tolist())) != len(live):
        raise ValueError("two rows name the same slot")
    new = _as_f64(pool).copy()
    N, H, dv = v.shape
    o = np.zeros((N, H, dv), dtype=np.float64)
    if len(live):
        sel = torch.as_tensor(live)
        cu = torch.arange(len(live) + 1, dtype=torch.int64)
        o_live, S = recurrent(q[sel], k[sel], v[sel], g[sel], scale, h0=new[idx[live]],
                              cu_seqlens=cu)
        o[live] = o_live
        new[idx[live]] = round_bf16(S) if storage == "bf16" else S
    return o, new


# ----------------------------------------------------------------------------------------
# the gated delta rule (GDN), numpy fp64


def gdn_recurrent(q, k, v, g, beta, scale, h0=None, cu_seqlens=None):
    """Token-by-token gated delta rule, fp64.

    "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules", section 1.1: per
    token the state decays by exp(g), the memory read at the key, kv = k S, is replaced by the
    value: v_new = beta (v - kv), S <- S + k^T v_new, and o = scale q S. The decay is applied
    before the memory read (the chunked form of section 1.2, whose W carries exp(g), computes
    exactly this; see the pins). q, k: bf16 [T, H, dk] packed (with cu_seqlens) or [B, T, H,
    dk]; v [.., dv]; g, beta fp32 [.., H]; h0 [nseq, H, dk, dv] or None. Returns (o [T, H, dv],
    hT [nseq, H, dk, dv]) float64.
    """
    q, k, v, g, cu = _packed(q, k, v, g, cu_seqlens)
    bd = _as_f64(beta).reshape(g.shape)
    qd, kd, vd, gd = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(g)
    T, H, dk = qd.shape
    dv = vd.shape[-1]
    nseq = len(cu) - 1
    h0d = None if h0 is None else _as_f64(h0).reshape(nseq, H, dk, dv)
    o = np.zeros((T, H, dv))
    hT = np.zeros((nseq, H, dk, dv))
    for n in range(nseq):
        s, e = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S = np.zeros((dk, dv)) if h0d is None else h0d[n, h].copy()
            for t in range(s, e):
                S = np.exp(gd[t, h]) * S
                v_new = bd[t, h] * (vd[t, h] - kd[t, h] @ S)
                S = S + np.outer(kd[t, h], v_new)
                o[t, h] = scale * (qd[t, h] @ S)
            hT[n, h] = S
    return o, hT


def _gdn_chunk_one(q, k, v, g, beta, scale, S, C):
    """One sequence and head in the chunked form (UT transform), fp64: q, k [L, dk], v [L, dv],
    g, beta [L], S [dk, dv]. The steps of the GDN/KDA page's section 1.2 (formulas 11-17)."""
    L = q.shape[0]
    o = np.empty((L, v.shape[1]))
    for c0 in range(0, L, C):
        qi, ki, vi = q[c0:c0 + C], k[c0:c0 + C], v[c0:c0 + C]
        n = qi.shape[0]
        b = np.cumsum(g[c0:c0 + C])                         # chunk decay
        gamma = np.exp(np.tril(b[:, None] - b[None, :]))    # masked difference, then exp
        kb = ki * beta[c0:c0 + C, None]
        vb = vi * beta[c0:c0 + C, None]
        # formula 11: T = -(K_beta K^T * gamma).tril(-1), then row by row T[i, :i] += T[i, :] T[:, :i]
        Tm = -np.tril(kb @ ki.T * gamma, -1)
        for i in range(1, n):
            Tm[i, :i] = Tm[i, :i] + Tm[i, :] @ Tm[:, :i]
        Tm = Tm + np.eye(n)
        W = Tm @ (kb * np.exp(b)[:, None])                  # formula 12
        U = Tm @ vb                                         # formula 13
        new_v = U - W @ S                                   # formula 15
        o_inter = (qi * np.exp(b)[:, None]) @ S
        o_intra = np.tril(qi @ ki.T * gamma) @ new_v
        S = S * np.exp(b[-1]) + (ki * np.exp(b[-1] - b)[:, None]).T @ new_v   # formula 16
        o[c0:c0 + C] = scale * (o_inter + o_intra)          # formula 17
    return o, S


def gdn_chunkwise(q, k, v, g, beta, scale, h0=None, cu_seqlens=None, chunk: int = 64):
    """Chunked fp64 form of the gated delta rule; same arguments and results as
    :func:`gdn_recurrent`."""
    q, k, v, g, cu = _packed(q, k, v, g, cu_seqlens)
    bd = _as_f64(beta).reshape(g.shape)
    qd, kd, vd, gd = _as_f64(q), _as_f64(k), _as_f64(v), _as_f64(g)
    T, H, dk = qd.shape
    dv = vd.shape[-1]
    nseq = len(cu) - 1
    h0d = None if h0 is None else _as_f64(h0).reshape(nseq, H, dk, dv)
    o = np.zeros((T, H, dv))
    hT = np.zeros((nseq, H, dk, dv))
    for n in range(nseq):
        s, e = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            S0 = np.zeros((dk, dv)) if h0d is None else h0d[n, h].copy()
            if e > s:
                o[s:e, h], hT[n, h] = _gdn_chunk_one(qd[s:e, h], kd[s:e, h], vd[s:e, h],
                                                     gd[s:e, h], bd[s:e, h], scale, S0, chunk)
            else:
                hT[n, h] = S0
    return o, hT


# ----------------------------------------------------------------------------------------
# q/k prologue: per-head RMSNorm and RoPE (numpy)


def rope_inv_freq(theta: float = 10000.0, d: int = 128) -> np.ndarray:
    """inv_freq[i] = theta^(-2i/d) for i < d/2, rounded to float32 (the RoPE of the Blueprint is
    computed on float32 values: "RoPE(q.float(), k.float(), pos)")."""
    return (theta ** (-np.arange(d // 2, dtype=np.float64) * 2.0 / d)).astype(np.float32)


def qk_prologue(x, w, pos, eps: float = 1e-6, theta: float = 10000.0) -> np.ndarray:
    """The q/k prologue of a lightning layer on head vectors x [..., 128].

    "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)": q =
    RMSNorm(q, w = [128]) per head (the page's RMSNorm: x / sqrt(mean(x^2) + eps) times the
    weight), in the model's bf16; then q = RoPE(q.float(), pos).bf16() with theta = 10000. The
    rotation pairs element i with i + 64 (rotate-half) by the angle pos * inv_freq[i]; the
    angle is the float32 product of float32 values, as a float32 RoPE computes it, and the
    rest is float64. x: bf16/float values [..., 128]; w: [128]; pos: integer positions,
    broadcast against x's leading shape. Returns float64 values that are bfloat16 numbers.
    """
    xd = _as_f64(x)
    wd = _as_f64(w).reshape(-1)
    d = xd.shape[-1]
    rms = np.sqrt((xd * xd).sum(axis=-1, keepdims=True) / d + eps)
    y = round_bf16(xd / rms * wd)
    pos32 = np.asarray(pos, dtype=np.float32)[..., None]
    ang = (pos32 * rope_inv_freq(theta, d)).astype(np.float64)      # float32 product
    c, s = np.cos(ang), np.sin(ang)
    h = d // 2
    lo, hi = y[..., :h], y[..., h:]
    return round_bf16(np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1))


# ----------------------------------------------------------------------------------------
# output norm and gate (numpy, fp64)


def output_norm_gate(o, z, w, eps: float = 1e-6) -> np.ndarray:
    """Per token: RMSNorm over all its features, times the weight, times sigmoid(z), fp64.

    "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)", block
    "Output Norm + Gate + Projection": o = RMSNorm(o, w) over the 4096 features of a token,
    then o * sigmoid(z) with z = h W_z^T; RMSNorm as the page's input_layernorm block gives
    it: rms = sqrt(sum of squares / n + eps), x / rms, times the weight element-wise.

    o, z: [T, F] (or [T, H, 128], flattened per token); w: [F]. Returns [T, F] float64.
    """
    od = _as_f64(o)
    od = od.reshape(od.shape[0], -1)
    zd = _as_f64(z).reshape(od.shape)
    wd = _as_f64(w).reshape(-1)
    rms = np.sqrt((od * od).sum(axis=1) / od.shape[1] + eps)
    return od / rms[:, None] * wd[None, :] * (1.0 / (1.0 + np.exp(-zd)))


def rel_fro(x, ref) -> float:
    """Relative Frobenius error ||x - ref||_F / ||ref||_F (fp64)."""
    x = _as_f64(x)
    ref = _as_f64(ref)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((x - ref).ravel())
    if den == 0.0:
        return float(num)
    return float(num / den)


def rel_fro_slices(x, ref, bounds) -> np.ndarray:
    """Relative Frobenius error of every (slice, head) block.

    ``x`` and ``ref`` are [R, H, ...] (rows, heads, then anything); ``bounds`` lists the row
    ranges (start, end) of the slices: the token ranges of the sequences for an output
    [T, H, d], or (n, n + 1) for each sequence of a state [N, H, d, d]. Returns a
    [len(bounds), H] array whose entry (i, h) is :func:`rel_fro` of x[s:e, h] against
    ref[s:e, h]. The tolerances are stated per sequence and head (each (sequence, head)
    pair runs its own recurrence), so the largest entry is what a parity test bounds.
    """
    x = _as_f64(x)
    ref = _as_f64(ref)
    if x.shape != ref.shape:
        raise ValueError(f"shape mismatch {x.shape} vs {ref.shape}")
    out = np.zeros((len(bounds), ref.shape[1]))
    for i, (s, e) in enumerate(bounds):
        for h in range(ref.shape[1]):
            out[i, h] = rel_fro(x[s:e, h], ref[s:e, h])
    return out


def seq_bounds(cu_seqlens, T: int | None = None):
    """Token ranges of the sequences: from ``cu_seqlens`` ([N+1] offsets), or one range
    [0, T) when it is None."""
    if cu_seqlens is None:
        return [(0, int(T))]
    cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    return list(zip(cu[:-1], cu[1:]))

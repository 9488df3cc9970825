"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each pin is independent of the oracle's own code path: closed forms, the quadratic
(parenthesised-the-other-way) form, printed values, special cases that reduce to plain
linear algebra, and invariants of the recurrence. Shapes use d_k != d_v wherever possible so
that a transposed state or operand cannot pass.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16(x):
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def _rand_case(T, H, dk, dv, seed, g_lo=-0.5, g_hi=0.0, nseq_lens=None, h0=True):
    """Small random packed case in the oracle's input format."""
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((T, H, dk), generator=gen).to(torch.bfloat16)
    k = torch.randn((T, H, dk), generator=gen).to(torch.bfloat16)
    v = torch.randn((T, H, dv), generator=gen).to(torch.bfloat16)
    g = g_lo + (g_hi - g_lo) * torch.rand((T, H), generator=gen)
    lens = nseq_lens or [T]
    assert sum(lens) == T
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    hz = torch.randn((len(lens), H, dk, dv), generator=gen) * 0.5 if h0 else None
    return q, k, v, g.float(), hz, cu


def _read_table(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


# ---------------------------------------------------------------------------------------
# (QK)V = Q(KV): with g = 0 the recurrence equals masked causal attention without softmax
# ("MiniCPM-SALA — Complete Blueprint", "Why Not Just Use Linear Attention Everywhere?").


@pytest.mark.parametrize("T,H,dk,dv", [(1, 1, 3, 5), (37, 2, 5, 3), (200, 1, 128, 128)])
def test_associativity_g_zero(T, H, dk, dv):
    q, k, v, _, _, cu = _rand_case(T, H, dk, dv, seed=T + dk)
    g = torch.zeros((T, H))
    scale = 0.37
    o, hT = oracle.recurrent(q, k, v, g, scale, cu_seqlens=cu)
    qd, kd, vd = (x.double().numpy() for x in (q, k, v))
    for h in range(H):
        # (Q K^T masked to j <= t) V, evaluated with numpy: the other parenthesisation
        A = np.tril(qd[:, h] @ kd[:, h].T)
        ref = scale * (A @ vd[:, h])
        assert oracle.rel_fro(o[:, h], ref) < 1e-12
        # K^T V is the state after all tokens
        assert oracle.rel_fro(hT[0, h], kd[:, h].T @ vd[:, h]) < 1e-12


# ---------------------------------------------------------------------------------------
# Unrolled closed form for a constant per-head alpha ("MiniCPM-SALA — Complete Blueprint",
# "Why Linear Attention Loses Information", Problem 1):
#   S_n = alpha^n S_0 + sum_{i=1..n} alpha^(n-i) k_i^T v_i


@pytest.mark.parametrize("n,dk,dv", [(1, 4, 6), (50, 4, 6), (300, 7, 2)])
def test_closed_form_constant_alpha(n, dk, dv):
    H = 3
    alphas = [0.40, 0.80, 0.999]
    q, k, v, _, h0, cu = _rand_case(n, H, dk, dv, seed=n)
    g = torch.tensor([math.log(a) for a in alphas], dtype=torch.float32).expand(n, H).contiguous()
    _, hT = oracle.recurrent(q, k, v, g, 1.0, h0=h0, cu_seqlens=cu)
    kd, vd = k.double().numpy(), v.double().numpy()
    for h in range(H):
        a = math.exp(float(g[0, h]))       # the alpha the oracle sees (fp32 log-decay)
        ref = a ** n * h0[0, h].double().numpy()
        for i in range(1, n + 1):
            ref = ref + a ** (n - i) * np.outer(kd[i - 1, h], vd[i - 1, h])
        assert oracle.rel_fro(hT[0, h], ref) < 1e-12


# ---------------------------------------------------------------------------------------
# Printed decay values.


def _decay_after(alpha, n):
    """alpha^n as the oracle's state decay sees it: k = v = 0, h0 = 1, n tokens of g = ln alpha."""
    one = torch.zeros((n, 1, 1), dtype=torch.bfloat16)
    g = torch.full((n, 1), math.log(alpha), dtype=torch.float32)
    h0 = torch.ones((1, 1, 1, 1), dtype=torch.float64)
    _, hT = oracle.recurrent(one, one, one, g, 1.0, h0=h0)
    return float(hT[0, 0, 0, 0])


def test_decay_over_distance_table():
    rows = _read_table("decay_over_distance.txt")
    assert len(rows) == 18
    for alpha_s, n_s, printed_s, check in rows:
        alpha, n, printed = float(alpha_s), int(n_s), float(printed_s)
        got = _decay_after(alpha, n)
        if check == "zero":
            assert 0.0 <= got < 1e-6, (alpha, n, got)
        elif check == "rel1pct":
            assert abs(got - printed) <= 0.01 * printed, (alpha, n, got)
        else:
            mant = printed_s.lower().split("e")[0]
            exp10 = int(printed_s.lower().split("e")[1]) if "e" in printed_s.lower() else 0
            decimals = len(mant.split(".")[1]) if "." in mant else 0
            half_ulp = 0.5 * 10.0 ** (exp10 - decimals)
            assert abs(got - printed) <= half_ulp, (alpha, n, got, printed)


def test_per_head_decay_printed():
    for g_s, alpha_s in _read_table("per_head_decay.txt"):
        one = torch.zeros((1, 1, 1), dtype=torch.bfloat16)
        g = torch.full((1, 1), float(g_s), dtype=torch.float32)
        _, hT = oracle.recurrent(one, one, one, g, 1.0, h0=torch.ones((1, 1, 1, 1)))
        decimals = len(alpha_s.split(".")[1])
        assert abs(float(hT.ravel()[0]) - float(alpha_s)) <= 0.5 * 10.0 ** -decimals


def test_scale_constant():
    rows = dict((r[0], r[1]) for r in _read_table("constants.txt"))
    from gated_linear_attention_gb300 import inputs
    assert int(rows["head_dim"]) == inputs.D
    assert abs(inputs.SCALE - float(rows["attn_scale"])) <= 0.5e-5


# ---------------------------------------------------------------------------------------
# Special case: k = v = 0 leaves only the initial state, decayed:
#   o_t = scale * exp(G_t) q_t h0,  hT = exp(G_T) h0.


def test_h0_only_path():
    T, H, dk, dv = 70, 2, 6, 4
    q, _, _, g, h0, cu = _rand_case(T, H, dk, dv, seed=5, g_lo=-0.3)
    z = torch.zeros((T, H, dk), dtype=torch.bfloat16)
    zv = torch.zeros((T, H, dv), dtype=torch.bfloat16)
    o, hT = oracle.recurrent(q, z, zv, g, 0.25, h0=h0, cu_seqlens=cu)
    G = np.cumsum(g.double().numpy(), axis=0)          # [T, H]
    qd = q.double().numpy()
    for h in range(H):
        H0 = h0[0, h].double().numpy()
        ref_o = 0.25 * np.exp(G[:, h])[:, None] * (qd[:, h] @ H0)
        assert oracle.rel_fro(o[:, h], ref_o) < 1e-13
        assert oracle.rel_fro(hT[0, h], math.exp(G[-1, h]) * H0) < 1e-13


# ---------------------------------------------------------------------------------------
# The quadratic form with per-token decay and a nonzero h0 (brute force, tiny sizes).


@pytest.mark.parametrize("lens,H,dk,dv", [([1], 1, 2, 3), ([5, 0, 12], 2, 3, 5),
                                           ([33, 64, 1], 3, 8, 4), ([130], 1, 16, 16)])
def test_recurrent_vs_bruteforce(lens, H, dk, dv):
    T = sum(lens)
    q, k, v, g, h0, cu = _rand_case(T, H, dk, dv, seed=T + H, g_lo=-1.0, nseq_lens=lens)
    o, hT = oracle.recurrent(q, k, v, g, 0.3, h0=h0, cu_seqlens=cu)
    ob, hb = oracle.bruteforce(q, k, v, g, 0.3, h0=h0, cu_seqlens=cu)
    assert oracle.rel_fro(o, ob) < 1e-12
    assert oracle.rel_fro(hT, hb) < 1e-12


# ---------------------------------------------------------------------------------------
# Chunked form (its own code path, following the GDN/KDA page's chunk recipe) against the
# recurrence: the two forms compute the same thing.


@pytest.mark.parametrize("lens,chunk", [([1], 64), ([63], 64), ([64], 64), ([65], 64),
                                        ([127, 200, 0, 3], 64), ([300], 16)])
def test_chunkwise_vs_recurrent(lens, chunk):
    T, H, dk, dv = sum(lens), 2, 12, 20
    q, k, v, g, h0, cu = _rand_case(T, H, dk, dv, seed=7 + T, g_lo=-0.9, nseq_lens=lens)
    o, hT = oracle.recurrent(q, k, v, g, 0.125, h0=h0, cu_seqlens=cu)
    oc, hc = oracle.chunkwise(q, k, v, g, 0.125, h0=h0, cu_seqlens=cu, chunk=chunk)
    assert oracle.rel_fro(oc, o) < 1e-10
    assert oracle.rel_fro(hc, hT) < 1e-10


def test_chunkwise_vs_recurrent_full_dim():
    T, H = 200, 2
    q, k, v, g, h0, cu = _rand_case(T, H, 128, 128, seed=11, g_lo=-0.2)
    o, hT = oracle.recurrent(q, k, v, g, 128 ** -0.5, h0=h0, cu_seqlens=cu)
    oc, hc = oracle.chunkwise(q, k, v, g, 128 ** -0.5, h0=h0, cu_seqlens=cu)
    assert oracle.rel_fro(oc, o) < 1e-10
    assert oracle.rel_fro(hc, hT) < 1e-10


# ---------------------------------------------------------------------------------------
# Invariants: the state is the whole memory of the past (fixed size regardless of T), so a
# sequence split in two calls chained through hT -> h0 equals one call; packed varlen equals
# separate calls; a zero-length sequence returns h0.


def test_split_resume():
    T, H, dk, dv = 150, 2, 8, 6
    q, k, v, g, h0, cu = _rand_case(T, H, dk, dv, seed=3, g_lo=-0.4)
    o, hT = oracle.recurrent(q, k, v, g, 0.5, h0=h0, cu_seqlens=cu)
    for cut in (0, 1, 64, 97, 150):
        o1, h1 = oracle.recurrent(q[:cut], k[:cut], v[:cut], g[:cut], 0.5, h0=h0,
                                  cu_seqlens=torch.tensor([0, cut]))
        o2, h2 = oracle.recurrent(q[cut:], k[cut:], v[cut:], g[cut:], 0.5, h0=h1,
                                  cu_seqlens=torch.tensor([0, T - cut]))
        np.testing.assert_allclose(np.concatenate([o1, o2]), o, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(h2, hT, rtol=1e-12, atol=1e-14)


def test_varlen_equals_separate_calls():
    lens = [17, 0, 64, 5]
    T, H, dk, dv = sum(lens), 3, 4, 4
    q, k, v, g, h0, cu = _rand_case(T, H, dk, dv, seed=9, nseq_lens=lens)
    o, hT = oracle.recurrent(q, k, v, g, 0.7, h0=h0, cu_seqlens=cu)
    for n, (s, e) in enumerate(zip(cu[:-1].tolist(), cu[1:].tolist())):
        on, hn = oracle.recurrent(q[s:e], k[s:e], v[s:e], g[s:e], 0.7, h0=h0[n:n + 1],
                                  cu_seqlens=torch.tensor([0, e - s]))
        np.testing.assert_array_equal(on, o[s:e])
        np.testing.assert_array_equal(hn[0], hT[n])
    # the empty sequence keeps its initial state exactly
    np.testing.assert_array_equal(hT[1], h0[1].double().numpy())


def test_head_subset_matches_all_heads():
    T, H = 40, 5
    q, k, v, g, h0, cu = _rand_case(T, H, 8, 8, seed=2)
    o, hT = oracle.recurrent(q, k, v, g, 0.2, h0=h0, cu_seqlens=cu)
    heads = [4, 0, 2]
    os_, hs = oracle.recurrent(q, k, v, g, 0.2, h0=h0, cu_seqlens=cu, heads=heads)
    np.testing.assert_array_equal(os_, o[:, heads])
    np.testing.assert_array_equal(hs, hT[:, heads])


def test_decode_steps_equal_prefill():
    """N one-token steps carried through the state equal one pass over the N tokens."""
    T, H, dk, dv = 25, 2, 6, 5
    q, k, v, g, h0, cu = _rand_case(T, H, dk, dv, seed=13)
    o, hT = oracle.recurrent(q, k, v, g, 0.9, h0=h0, cu_seqlens=cu)
    S = h0
    for t in range(T):
        ot, S = oracle.recurrent(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], 0.9, h0=S,
                                 cu_seqlens=torch.tensor([0, 1]))
        np.testing.assert_allclose(ot[0], o[t], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S, hT, rtol=1e-13, atol=1e-15)


def test_bf16_inputs_read_exactly():
    """The oracle reads bf16 bit patterns exactly (no re-rounding): with one token, h0 = 0 and
    g = 0, o = scale (q . k) v and hT = k^T v in fp64 from the bf16 values."""
    vals = torch.tensor([[1.0 + 2 ** -7, -3.0, 2 ** -20]], dtype=torch.float32)
    q = vals.to(torch.bfloat16).reshape(1, 1, 3)
    k = torch.tensor([[0.5, 0.25, -1.0 - 2 ** -7]]).to(torch.bfloat16).reshape(1, 1, 3)
    v = torch.tensor([[7.0, -2 ** -9]]).to(torch.bfloat16).reshape(1, 1, 2)
    g = torch.zeros((1, 1))
    o, hT = oracle.recurrent(q, k, v, g, 1.0)
    qd, kd, vd = q.double().numpy()[0, 0], k.double().numpy()[0, 0], v.double().numpy()[0, 0]
    assert o[0, 0, 0] == float(np.dot(qd, kd)) * vd[0]
    np.testing.assert_array_equal(hT[0, 0], np.outer(kd, vd))


def test_oracle_rejects_bad_arguments():
    q = torch.zeros((4, 1, 2), dtype=torch.bfloat16)
    g = torch.zeros((4, 1))
    with pytest.raises(ValueError):
        oracle.recurrent(q, q, q, g, 1.0, cu_seqlens=torch.tensor([0, 3, 2]))
    with pytest.raises(ValueError):
        oracle.recurrent(q, q, q, g, 1.0, heads=[1])


# ---------------------------------------------------------------------------------------
# one decode step on pooled states ("MiniCPM-SALA — Complete Blueprint", "Memory
# Architecture": per-request temporal states in a per-layer pool, loaded, updated and saved
# back in place; 1 MB per request in bf16 for 32 heads)


def _pool_case(N, H, dk, dv, P, seed, pad=()):
    gen = torch.Generator().manual_seed(seed)
    q = torch.randn((N, H, dk), generator=gen).to(torch.bfloat16)
    k = torch.randn((N, H, dk), generator=gen).to(torch.bfloat16)
    v = torch.randn((N, H, dv), generator=gen).to(torch.bfloat16)
    g = -0.5 * torch.rand((N, H), generator=gen)
    pool = torch.randn((P, H, dk, dv), generator=gen) * 0.5
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32)
    for n in pad:
        idx[n] = -1
    return q, k, v, g, pool, idx


def _pool_step_numpy(q, k, v, g, scale, pool, idx):
    """The step written out per row with numpy outer products (no oracle code)."""
    new = pool.double().numpy().copy()
    N, H, _ = q.shape
    o = np.zeros((N, H, v.shape[-1]))
    for n in range(N):
        i = int(idx[n])
        if i < 0:
            continue
        for h in range(H):
            S = math.exp(float(g[n, h])) * new[i, h] + np.outer(k[n, h].double().numpy(),
                                                                v[n, h].double().numpy())
            o[n, h] = scale * (q[n, h].double().numpy() @ S)
            new[i, h] = S
    return o, new


def test_pool_step_matches_outer_product_restatement():
    q, k, v, g, pool, idx = _pool_case(N=5, H=3, dk=7, dv=4, P=9, seed=41, pad=(2,))
    o, new = oracle.recurrent_step_indexed(q, k, v, g, 0.61, pool, idx)
    o_ref, new_ref = _pool_step_numpy(q, k, v, g, 0.61, pool, idx)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(new, new_ref, rtol=1e-12, atol=1e-12)
    # the padding row reads nothing and writes zeros; slots nobody names are untouched
    assert np.all(o[2] == 0.0)
    named = set(int(i) for i in idx if i >= 0)
    for i in range(9):
        if i not in named:
            assert np.array_equal(new[i], pool[i].double().numpy())


def test_pool_step_permutation_invariance():
    # relabelling the pool's slots (and the indices with them) changes nothing else
    q, k, v, g, pool, idx = _pool_case(N=4, H=2, dk=5, dv=6, P=7, seed=42, pad=(1,))
    perm = torch.randperm(7, generator=torch.Generator().manual_seed(7))
    inv = torch.argsort(perm)
    o1, new1 = oracle.recurrent_step_indexed(q, k, v, g, 0.3, pool, idx)
    idx2 = torch.where(idx >= 0, inv[idx.clamp(min=0).long()].to(torch.int32), idx)
    o2, new2 = oracle.recurrent_step_indexed(q, k, v, g, 0.3, pool[perm], idx2)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(new1[perm.numpy()], new2)


def test_round_bf16_matches_library_rounding():
    # on values exactly representable in float32, rounding to bfloat16 directly equals
    # torch's float32 -> bfloat16 conversion (round to nearest even)
    x = np.random.default_rng(5).standard_normal(200000).astype(np.float32)
    x = np.concatenate([x, x * 1e-20, x * 1e20, np.float32([0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8])])
    want = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x.astype(np.float64)), want)
    # ties go to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert oracle.round_bf16(1.0 + 2 ** -8) == 1.0
    assert oracle.round_bf16(1.0 + 3 * 2 ** -8) == 1.0 + 2 ** -6


def test_pool_step_bf16_storage():
    q, k, v, g, pool32, idx = _pool_case(N=4, H=2, dk=6, dv=5, P=6, seed=43, pad=(0,))
    pool = pool32.to(torch.bfloat16)
    o, new = oracle.recurrent_step_indexed(q, k, v, g, 0.5, pool, idx, storage="bf16")
    o_ref, S_ref = _pool_step_numpy(q, k, v, g, 0.5, pool.float(), idx)
    # o reads the updated state before rounding
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
    # stored values are bfloat16 numbers within half a unit in the last place of the state
    assert np.array_equal(torch.from_numpy(new).to(torch.bfloat16).double().numpy(), new)
    live = [int(i) for i in idx if i >= 0]
    err = np.abs(new[live] - S_ref[live])
    assert np.all(err <= np.abs(S_ref[live]) * 2.0 ** -8)
    # the slot of the padding row is untouched
    pad_slot = [i for i in range(6) if i not in live]
    np.testing.assert_array_equal(new[pad_slot], pool[pad_slot].double().numpy())


def test_pool_step_rejects_bad_indices():
    q, k, v, g, pool, idx = _pool_case(N=3, H=1, dk=4, dv=4, P=5, seed=44)
    with pytest.raises(ValueError):
        oracle.recurrent_step_indexed(q, k, v, g, 0.5, pool, torch.tensor([0, 5, 1], dtype=torch.int32))
    with pytest.raises(ValueError):
        oracle.recurrent_step_indexed(q, k, v, g, 0.5, pool, torch.tensor([2, 2, 1], dtype=torch.int32))


# ---------------------------------------------------------------------------------------
# output norm and gate ("MiniCPM-SALA — Complete Blueprint", "Output Norm + Gate +
# Projection": RMSNorm over the token's 4096 features with a weight, times sigmoid(z))


def test_output_gate_matches_library_rms_norm_and_sigmoid():
    gen = torch.Generator().manual_seed(51)
    o = torch.randn((9, 3, 128), generator=gen, dtype=torch.float64)
    z = 3 * torch.randn((9, 3, 128), generator=gen, dtype=torch.float64)
    w = 1 + 0.2 * torch.randn(384, generator=gen, dtype=torch.float64)
    got = oracle.output_norm_gate(o, z, w, eps=1e-6)
    want = (torch.nn.functional.rms_norm(o.reshape(9, 384), (384,), w, eps=1e-6) *
            torch.sigmoid(z.reshape(9, 384))).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)


def test_output_gate_special_cases():
    F = 256
    # a constant row normalises to +-1 (up to eps); z = 0 halves it; w scales per feature
    o = np.full((1, F), 3.0)
    w = np.linspace(0.5, 1.5, F)
    got = oracle.output_norm_gate(o, np.zeros((1, F)), w, eps=0.0)
    np.testing.assert_allclose(got[0], 0.5 * w, rtol=1e-15)
    # a very open gate passes RMSNorm(o) * w through; a closed one gives zeros
    x = np.random.default_rng(3).standard_normal((2, F))
    rms = np.sqrt((x * x).mean(axis=1, keepdims=True))
    np.testing.assert_allclose(oracle.output_norm_gate(x, np.full((2, F), 60.0), w, eps=0.0),
                               x / rms * w, rtol=1e-12)
    assert np.all(np.abs(oracle.output_norm_gate(x, np.full((2, F), -80.0), w, eps=0.0)) < 1e-32)
    # scaling o by a > 0 changes nothing when eps = 0
    np.testing.assert_allclose(oracle.output_norm_gate(7.5 * x, x, w, eps=0.0),
                               oracle.output_norm_gate(x, x, w, eps=0.0), rtol=1e-13)
    # the page's printed epsilon: a zero row stays zero
    assert np.all(oracle.output_norm_gate(np.zeros((1, F)), x[:1], w, eps=1e-6) == 0.0)


# ---------------------------------------------------------------------------------------
# q/k prologue ("MiniCPM-SALA — Complete Blueprint", B2: QK RMSNorm per head with w = [128],
# then RoPE with theta = 10000 on float32 values, rounded to bf16)


def test_prologue_at_position_zero_is_rms_norm():
    gen = torch.Generator().manual_seed(61)
    x = torch.randn((5, 3, 128), generator=gen).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    got = oracle.qk_prologue(x, w, np.zeros((5, 1)), eps=1e-6)
    want = torch.nn.functional.rms_norm(x.double(), (128,), w.double(), eps=1e-6).numpy()
    np.testing.assert_array_equal(got, oracle.round_bf16(want))


def test_prologue_rotation_closed_form():
    # a head vector along element 0: after the norm it is sqrt(128) e_0 (w = 1); element i = 0
    # turns with element 64 by the angle pos * theta^0 = pos
    x = np.zeros((1, 128))
    x[0, 0] = 3.0
    for pos in (1, 2, 7):
        y = oracle.qk_prologue(x, np.ones(128), np.array([pos]), eps=0.0)[0]
        r = math.sqrt(128.0)
        assert abs(y[0] - r * math.cos(pos)) <= r * 2 ** -8
        assert abs(y[64] - r * math.sin(pos)) <= r * 2 ** -8
        assert np.all(y[1:64] == 0) and np.all(y[65:] == 0)
    # element i = 32 turns by pos * theta^(-1/2) = pos / 100
    x = np.zeros((1, 128))
    x[0, 32] = 1.0
    y = oracle.qk_prologue(x, np.ones(128), np.array([50]), eps=0.0)[0]
    assert abs(y[32] - math.sqrt(128) * math.cos(0.5)) <= math.sqrt(128) * 2 ** -8
    assert abs(y[96] - math.sqrt(128) * math.sin(0.5)) <= math.sqrt(128) * 2 ** -8


def test_prologue_rotation_invariants():
    gen = torch.Generator().manual_seed(62)
    q = torch.randn((1, 128), generator=gen).to(torch.bfloat16)
    k = torch.randn((1, 128), generator=gen).to(torch.bfloat16)
    w = np.ones(128)
    y0 = oracle.qk_prologue(q, w, np.array([0]))[0]
    y = oracle.qk_prologue(q, w, np.array([37]))[0]
    # each (i, i + 64) pair keeps its length (to the bf16 rounding)
    n0 = np.hypot(y0[:64], y0[64:])
    n1 = np.hypot(y[:64], y[64:])
    np.testing.assert_allclose(n1, n0, rtol=2 ** -6, atol=1e-3)
    # q . k depends on the positions' difference only
    dots = []
    for m, n in ((10, 3), (17, 10), (107, 100)):
        a = oracle.qk_prologue(q, w, np.array([m]))[0]
        b = oracle.qk_prologue(k, w, np.array([n]))[0]
        dots.append(a @ b)
    assert max(dots) - min(dots) <= 0.02 * abs(dots[0]) + 0.05


# ---------------------------------------------------------------------------------------
# gated delta rule ("Formulas and Code for Adapting Inference to GDN/KDA Linear Modules":
# recurrent form, section 1.1; chunked form with the UT transform, section 1.2)


def _gdn_case(T, H, dk, dv, seed, lens=None, h0=True):
    gen = torch.Generator().manual_seed(seed)
    q = torch.nn.functional.normalize(torch.randn((T, H, dk), generator=gen), dim=-1).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn((T, H, dk), generator=gen), dim=-1).to(torch.bfloat16)
    v = torch.randn((T, H, dv), generator=gen).to(torch.bfloat16)
    g = -0.4 * torch.rand((T, H), generator=gen)
    beta = torch.rand((T, H), generator=gen)
    lens = lens or [T]
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int64)
    hz = torch.randn((len(lens), H, dk, dv), generator=gen) * 0.3 if h0 else None
    return q, k, v, g, beta, hz, cu


@pytest.mark.parametrize("lens,chunk", [([37], 8), ([130, 0, 64, 5], 16), ([200], 64)])
def test_gdn_chunked_form_equals_recurrence(lens, chunk):
    # the page's chunked form (UT transform, W carrying exp(g)) reaches the recurrence with
    # the decay applied before the memory read
    q, k, v, g, beta, h0, cu = _gdn_case(sum(lens), 2, 12, 7, seed=sum(lens), lens=lens)
    o1, h1 = oracle.gdn_recurrent(q, k, v, g, beta, 0.7, h0=h0, cu_seqlens=cu)
    o2, h2 = oracle.gdn_chunkwise(q, k, v, g, beta, 0.7, h0=h0, cu_seqlens=cu, chunk=chunk)
    assert oracle.rel_fro(o2, o1) < 1e-12
    assert oracle.rel_fro(h2, h1) < 1e-12


def test_gdn_delta_rule_retrieval():
    # g = 0, beta = 1, unit-norm key: after the write, reading at that key returns its value
    dk, dv = 16, 9
    rng = np.random.default_rng(4)
    S0 = rng.standard_normal((1, 1, dk, dv))
    kk = rng.standard_normal(dk)
    kk /= np.linalg.norm(kk)
    vv = rng.standard_normal(dv)
    k = torch.tensor(kk, dtype=torch.float64).reshape(1, 1, dk)
    v = torch.tensor(vv, dtype=torch.float64).reshape(1, 1, dv)
    _, hT = oracle.gdn_recurrent(k, k, v, torch.zeros((1, 1)), torch.ones((1, 1)), 1.0, h0=S0,
                                 cu_seqlens=torch.tensor([0, 1]))
    np.testing.assert_allclose(kk @ hT[0, 0], vv, rtol=1e-12, atol=1e-12)


def test_gdn_beta_zero_only_decays():
    q, k, v, g, beta, h0, cu = _gdn_case(40, 2, 8, 6, seed=5)
    o, hT = oracle.gdn_recurrent(q, k, v, g, torch.zeros_like(beta), 0.5, h0=h0, cu_seqlens=cu)
    G = np.cumsum(g.double().numpy(), axis=0)
    for h in range(2):
        want_o = 0.5 * np.exp(G[:, h])[:, None] * (q[:, h].double().numpy() @ h0[0, h].double().numpy())
        np.testing.assert_allclose(o[:, h], want_o, rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(hT[0, h], np.exp(G[-1, h]) * h0[0, h].double().numpy(), rtol=1e-12)


def test_gdn_orthogonal_keys_reduce_to_simple_gla():
    # keys along distinct coordinate axes never read back what an earlier token wrote, so
    # with beta = 1 and no initial state the gated delta rule is Simple GLA
    T, H, dk, dv = 20, 1, 24, 5
    gen = torch.Generator().manual_seed(8)
    k = torch.zeros((T, H, dk))
    k[torch.arange(T), 0, torch.arange(T)] = 1.0
    k = k.to(torch.bfloat16)
    q = torch.randn((T, H, dk), generator=gen).to(torch.bfloat16)
    v = torch.randn((T, H, dv), generator=gen).to(torch.bfloat16)
    g = -0.3 * torch.rand((T, H), generator=gen)
    cu = torch.tensor([0, T])
    o1, h1 = oracle.gdn_recurrent(q, k, v, g, torch.ones((T, H)), 0.9, cu_seqlens=cu)
    o2, h2 = oracle.recurrent(q, k, v, g, 0.9, cu_seqlens=cu)
    assert oracle.rel_fro(o1, o2) < 1e-12 and oracle.rel_fro(h1, h2) < 1e-12

"""The pins of the oracle's numpy functions are strong enough: plausible mistakes planted in a
copy of each function (a text substitution of its source, executed in the oracle module's
namespace, on the CPU) each fail at least one of the checks the pins make.

The committed oracle carries no mutation code.
"""
import inspect
import math

import numpy as np
import pytest
import torch

import oracle


def _mutant(fn, old, new, extra=()):
    """fn's source with `old` replaced by `new`, compiled in the oracle's namespace (extra:
    other functions of the module that the mutant should see in mutated form)."""
    src = inspect.getsource(fn)
    assert src.count(old) == 1, (fn.__name__, old)
    ns = dict(vars(oracle))
    for name, f in extra:
        ns[name] = f
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns[fn.__name__]


# ---------------------------------------------------------------------------------------
# gated delta rule


def _gdn_case(T=40, H=2, dk=12, dv=7, seed=3):
    gen = torch.Generator().manual_seed(seed)
    q = torch.nn.functional.normalize(torch.randn((T, H, dk), generator=gen), dim=-1).to(torch.bfloat16)
    k = torch.nn.functional.normalize(torch.randn((T, H, dk), generator=gen), dim=-1).to(torch.bfloat16)
    v = torch.randn((T, H, dv), generator=gen).to(torch.bfloat16)
    g = -0.4 * torch.rand((T, H), generator=gen)
    beta = torch.rand((T, H), generator=gen)
    h0 = torch.randn((1, H, dk, dv), generator=gen) * 0.3
    return q, k, v, g, beta, h0, torch.tensor([0, T])


def _gdn_pins_hold(rec, chunked):
    """The GDN pins: chunked == recurrent; delta-rule retrieval; beta = 0 closed form;
    orthogonal keys reduce to Simple GLA."""
    q, k, v, g, beta, h0, cu = _gdn_case()
    o1, h1 = rec(q, k, v, g, beta, 0.7, h0=h0, cu_seqlens=cu)
    o2, h2 = chunked(q, k, v, g, beta, 0.7, h0=h0, cu_seqlens=cu, chunk=16)
    if not (oracle.rel_fro(o2, o1) < 1e-12 and oracle.rel_fro(h2, h1) < 1e-12):
        return False
    rng = np.random.default_rng(4)
    S0 = rng.standard_normal((1, 1, 16, 9))
    kk = rng.standard_normal(16)
    kk /= np.linalg.norm(kk)
    vv = rng.standard_normal(9)
    kt = torch.tensor(kk).reshape(1, 1, 16)
    _, hT = rec(kt, kt, torch.tensor(vv).reshape(1, 1, 9), torch.zeros((1, 1)), torch.ones((1, 1)),
                1.0, h0=S0, cu_seqlens=torch.tensor([0, 1]))
    if not np.allclose(kk @ hT[0, 0], vv, rtol=1e-12, atol=1e-12):
        return False
    o, hT = rec(q, k, v, g, torch.zeros_like(beta), 0.5, h0=h0, cu_seqlens=cu)
    G = np.cumsum(g.double().numpy(), axis=0)
    want = 0.5 * np.exp(G[:, 0])[:, None] * (q[:, 0].double().numpy() @ h0[0, 0].double().numpy())
    if not np.allclose(o[:, 0], want, rtol=1e-12, atol=1e-14):
        return False
    T = 20
    ko = torch.zeros((T, 1, 24))
    ko[torch.arange(T), 0, torch.arange(T)] = 1.0
    qo = torch.randn((T, 1, 24), generator=torch.Generator().manual_seed(8)).to(torch.bfloat16)
    vo = torch.randn((T, 1, 5), generator=torch.Generator().manual_seed(9)).to(torch.bfloat16)
    go = -0.3 * torch.rand((T, 1), generator=torch.Generator().manual_seed(10))
    a1, _ = rec(qo, ko.to(torch.bfloat16), vo, go, torch.ones((T, 1)), 0.9, cu_seqlens=torch.tensor([0, T]))
    a2, _ = oracle.recurrent(qo, ko.to(torch.bfloat16), vo, go, 0.9, cu_seqlens=torch.tensor([0, T]))
    return oracle.rel_fro(a1, a2) < 1e-12


GDN_REC_MUTANTS = {
    "read before decay": ("                S = np.exp(gd[t, h]) * S\n                v_new = bd[t, h] * (vd[t, h] - kd[t, h] @ S)\n                S = S + np.outer(kd[t, h], v_new)",
                          "                v_new = bd[t, h] * (vd[t, h] - kd[t, h] @ S)\n                S = np.exp(gd[t, h]) * S + np.outer(kd[t, h], v_new)"),
    "beta dropped": ("v_new = bd[t, h] * (vd[t, h] - kd[t, h] @ S)", "v_new = (vd[t, h] - kd[t, h] @ S)"),
    "memory read with the wrong sign": ("(vd[t, h] - kd[t, h] @ S)", "(vd[t, h] + kd[t, h] @ S)"),
    "memory read transposed": ("kd[t, h] @ S)", "(S @ vd[t, h])[:dv] * 0 + (S.T @ kd[t, h]) * 0 + S[0])"),
    "scale dropped": ("o[t, h] = scale * (qd[t, h] @ S)", "o[t, h] = (qd[t, h] @ S)"),
}

GDN_CHUNK_MUTANTS = {
    "T strict tril made inclusive": ("Tm = -np.tril(kb @ ki.T * gamma, -1)", "Tm = -np.tril(kb @ ki.T * gamma, 0)"),
    "identity not added": ("        Tm = Tm + np.eye(n)\n", ""),
    "W without the decay": ("W = Tm @ (kb * np.exp(b)[:, None])", "W = Tm @ kb"),
    "state carry without the end decay": ("(ki * np.exp(b[-1] - b)[:, None]).T @ new_v", "ki.T @ new_v"),
    "row recursion uses the wrong rows": ("Tm[i, :i] = Tm[i, :i] + Tm[i, :] @ Tm[:, :i]",
                                          "Tm[i, :i] = Tm[i, :i] + Tm[:, i] @ Tm[:, :i]"),
}


def test_gdn_pins_hold_for_the_committed_oracle():
    assert _gdn_pins_hold(oracle.gdn_recurrent, oracle.gdn_chunkwise)


@pytest.mark.parametrize("name", sorted(GDN_REC_MUTANTS))
def test_gdn_recurrent_mutant_is_caught(name):
    old, new = GDN_REC_MUTANTS[name]
    m = _mutant(oracle.gdn_recurrent, old, new)
    try:
        ok = _gdn_pins_hold(m, oracle.gdn_chunkwise)
    except Exception:
        ok = False
    assert not ok, name


@pytest.mark.parametrize("name", sorted(GDN_CHUNK_MUTANTS))
def test_gdn_chunked_mutant_is_caught(name):
    old, new = GDN_CHUNK_MUTANTS[name]
    one = _mutant(oracle._gdn_chunk_one, old, new)
    m = _mutant(oracle.gdn_chunkwise, "_gdn_chunk_one(", "_gdn_chunk_one(", extra=[("_gdn_chunk_one", one)])
    try:
        ok = _gdn_pins_hold(oracle.gdn_recurrent, m)
    except Exception:
        ok = False
    assert not ok, name


# ---------------------------------------------------------------------------------------
# output norm and gate


def _gate_pins_hold(fn):
    gen = torch.Generator().manual_seed(51)
    o = torch.randn((9, 3, 128), generator=gen, dtype=torch.float64)
    z = 3 * torch.randn((9, 3, 128), generator=gen, dtype=torch.float64)
    w = 1 + 0.2 * torch.randn(384, generator=gen, dtype=torch.float64)
    want = (torch.nn.functional.rms_norm(o.reshape(9, 384), (384,), w, eps=1e-6) *
            torch.sigmoid(z.reshape(9, 384))).numpy()
    if not np.allclose(fn(o, z, w, eps=1e-6), want, rtol=1e-12, atol=1e-14):
        return False
    F = 256
    x = np.random.default_rng(3).standard_normal((2, F))
    wv = np.linspace(0.5, 1.5, F)
    return np.allclose(fn(np.full((1, F), 3.0), np.zeros((1, F)), wv, eps=0.0)[0], 0.5 * wv, rtol=1e-15)


GATE_MUTANTS = {
    "sum instead of mean": ("(od * od).sum(axis=1) / od.shape[1] + eps", "(od * od).sum(axis=1) + eps"),
    "square root dropped": ("rms = np.sqrt(", "rms = (("),
    "gate not a sigmoid": ("(1.0 / (1.0 + np.exp(-zd)))", "zd"),
    "weight dropped": ("* wd[None, :] *", "*"),
}


def test_gate_pins_hold_for_the_committed_oracle():
    assert _gate_pins_hold(oracle.output_norm_gate)


@pytest.mark.parametrize("name", sorted(GATE_MUTANTS))
def test_gate_mutant_is_caught(name):
    old, new = GATE_MUTANTS[name]
    if name == "square root dropped":
        new_src = ("rms = ((od * od).sum(axis=1) / od.shape[1] + eps)", )
        m = _mutant(oracle.output_norm_gate, "rms = np.sqrt((od * od).sum(axis=1) / od.shape[1] + eps)",
                    new_src[0])
    else:
        m = _mutant(oracle.output_norm_gate, old, new)
    try:
        ok = _gate_pins_hold(m)
    except Exception:
        ok = False
    assert not ok, name


# ---------------------------------------------------------------------------------------
# q/k prologue


def _prologue_pins_hold(fn):
    gen = torch.Generator().manual_seed(61)
    x = torch.randn((5, 3, 128), generator=gen).to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    want = torch.nn.functional.rms_norm(x.double(), (128,), w.double(), eps=1e-6).numpy()
    if not np.array_equal(fn(x, w, np.zeros((5, 1)), eps=1e-6), oracle.round_bf16(want)):
        return False
    r = math.sqrt(128.0)
    x = np.zeros((1, 128))
    x[0, 0] = 3.0
    for pos in (1, 2, 7):
        y = fn(x, np.ones(128), np.array([pos]), eps=0.0)[0]
        if abs(y[0] - r * math.cos(pos)) > r * 2 ** -8 or abs(y[64] - r * math.sin(pos)) > r * 2 ** -8:
            return False
    x = np.zeros((1, 128))
    x[0, 32] = 1.0
    y = fn(x, np.ones(128), np.array([50]), eps=0.0)[0]
    return abs(y[32] - r * math.cos(0.5)) <= r * 2 ** -8 and abs(y[96] - r * math.sin(0.5)) <= r * 2 ** -8


PROLOGUE_MUTANTS = {
    "rotation sign": ("lo * c - hi * s, hi * c + lo * s", "lo * c + hi * s, hi * c - lo * s"),
    "adjacent pairs instead of halves": ("lo, hi = y[..., :h], y[..., h:]", "lo, hi = y[..., 0::2], y[..., 1::2]"),
    "weight dropped": ("y = round_bf16(xd / rms * wd)", "y = round_bf16(xd / rms)"),
    "sum instead of mean": ("(xd * xd).sum(axis=-1, keepdims=True) / d + eps", "(xd * xd).sum(axis=-1, keepdims=True) + eps"),
}


def test_prologue_pins_hold_for_the_committed_oracle():
    assert _prologue_pins_hold(oracle.qk_prologue)


@pytest.mark.parametrize("name", sorted(PROLOGUE_MUTANTS))
def test_prologue_mutant_is_caught(name):
    old, new = PROLOGUE_MUTANTS[name]
    m = _mutant(oracle.qk_prologue, old, new)
    try:
        ok = _prologue_pins_hold(m)
    except Exception:
        ok = False
    assert not ok, name


def test_inv_freq_mutant_is_caught():
    # theta^(-i/128) instead of theta^(-2i/128)
    f = _mutant(oracle.rope_inv_freq, "* 2.0 / d)", "* 1.0 / d)")
    m = _mutant(oracle.qk_prologue, "rope_inv_freq(theta, d)", "rope_inv_freq(theta, d)", extra=[("rope_inv_freq", f)])
    assert not _prologue_pins_hold(m)


# ---------------------------------------------------------------------------------------
# decode on pooled states


def _pool_pins_hold(fn):
    gen = torch.Generator().manual_seed(41)
    N, H, dk, dv, P = 5, 3, 7, 4, 9
    q = torch.randn((N, H, dk), generator=gen).to(torch.bfloat16)
    k = torch.randn((N, H, dk), generator=gen).to(torch.bfloat16)
    v = torch.randn((N, H, dv), generator=gen).to(torch.bfloat16)
    g = -0.5 * torch.rand((N, H), generator=gen)
    pool = torch.randn((P, H, dk, dv), generator=gen) * 0.5
    idx = torch.randperm(P, generator=gen)[:N].to(torch.int32)
    idx[2] = -1
    new = pool.double().numpy().copy()
    o_ref = np.zeros((N, H, dv))
    for n in range(N):
        i = int(idx[n])
        if i < 0:
            continue
        for h in range(H):
            S = math.exp(float(g[n, h])) * new[i, h] + np.outer(k[n, h].double().numpy(), v[n, h].double().numpy())
            o_ref[n, h] = 0.61 * (q[n, h].double().numpy() @ S)
            new[i, h] = S
    o, got = fn(q, k, v, g, 0.61, pool, idx)
    if not (np.allclose(o, o_ref, rtol=1e-12, atol=1e-12) and np.allclose(got, new, rtol=1e-12, atol=1e-12)):
        return False
    o, got = fn(q, k, v, g, 0.61, pool.to(torch.bfloat16), idx, storage="bf16")
    return bool(np.array_equal(torch.from_numpy(got).to(torch.bfloat16).double().numpy(), got))


POOL_MUTANTS = {
    "slots shifted": ("new[idx[live]] = round_bf16(S) if storage == \"bf16\" else S",
                      "new[(idx[live] + 1) % P] = round_bf16(S) if storage == \"bf16\" else S"),
    "bf16 storage not rounded": ("new[idx[live]] = round_bf16(S) if storage == \"bf16\" else S",
                                 "new[idx[live]] = S"),
    "padding rows computed": ("live = np.nonzero(idx >= 0)[0]", "live = np.nonzero(idx >= -1)[0]"),
}


def test_pool_pins_hold_for_the_committed_oracle():
    assert _pool_pins_hold(oracle.recurrent_step_indexed)


@pytest.mark.parametrize("name", sorted(POOL_MUTANTS))
def test_pool_mutant_is_caught(name):
    old, new = POOL_MUTANTS[name]
    m = _mutant(oracle.recurrent_step_indexed, old, new)
    try:
        ok = _pool_pins_hold(m)
    except Exception:
        ok = False
    assert not ok, name

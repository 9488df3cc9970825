"""Pins of the parity metric itself: the relative Frobenius error ||x - ref||_F / ||ref||_F
(the tolerance the GPU parity tests apply, per (sequence, head) slice) against values worked
out by hand, and the slicing against planted errors of known size. Mutants of both functions
(a swapped numerator and denominator, a missing square root, a norm over the wrong axis, a
slice bound off by one) each fail one of these checks.
"""
import inspect
import math

import numpy as np
import pytest
import torch

import oracle


def _pins_rel_fro(f):
    checks = [
        # ||(3, 4) - (0, 2)|| / ||(0, 2)|| = sqrt(9 + 4) / 2; with the arguments swapped the
        # denominator would be 5
        abs(f([3.0, 4.0], [0.0, 2.0]) - math.sqrt(13.0) / 2.0) < 1e-15,
        # a zero reference gives the absolute error
        abs(f([3.0, 4.0], [0.0, 0.0]) - 5.0) < 1e-15,
        # difference diag(3, 4): Frobenius 5 (spectral norm 4, largest row 4, sum of |.| 7)
        abs(f(np.array([[4.0, 0.0], [0.0, 4.0]]), np.array([[1.0, 0.0], [0.0, 0.0]])) - 5.0) < 1e-14,
        # exact agreement
        f(np.ones((3, 5)), np.ones((3, 5))) == 0.0,
        # bf16 input: 1 + 2^-7 is exactly representable, so the error is exactly 2^-7
        abs(f(torch.full((4,), 1.0 + 2.0 ** -7, dtype=torch.bfloat16), torch.ones(4)) - 2.0 ** -7) < 1e-15,
    ]
    return all(checks)


def _pins_slices(f):
    rng = np.random.default_rng(7)
    ref = rng.standard_normal((10, 3, 4))
    delta = np.zeros_like(ref)
    delta[3:10, 1] = rng.standard_normal((7, 4))
    bounds = [(0, 3), (3, 3), (3, 10)]
    out = f(ref + delta, ref, bounds)
    want = np.linalg.norm(delta[3:10, 1]) / np.linalg.norm(ref[3:10, 1])
    ok = out.shape == (3, 3) and abs(out[2, 1] - want) < 1e-14
    mask = np.ones_like(out, dtype=bool)
    mask[2, 1] = False
    ok = ok and np.all(out[mask] == 0.0)
    # an error confined to one row of a state [N, H, d, d]
    S = rng.standard_normal((4, 2, 3, 3))
    E = np.zeros_like(S)
    E[2, 0, 1, 1] = 0.5
    out2 = f(S + E, S, [(n, n + 1) for n in range(4)])
    ok = ok and abs(out2[2, 0] - 0.5 / np.linalg.norm(S[2, 0])) < 1e-14
    ok = ok and np.count_nonzero(out2) == 1
    return bool(ok)


def test_rel_fro_pins():
    assert _pins_rel_fro(oracle.rel_fro)


def test_rel_fro_slices_pins():
    assert _pins_slices(oracle.rel_fro_slices)


def test_seq_bounds():
    assert oracle.seq_bounds(torch.tensor([0, 5, 5, 12])) == [(0, 5), (5, 5), (5, 12)]
    assert oracle.seq_bounds(None, 9) == [(0, 9)]


def test_rel_fro_shape_mismatch_rejected():
    with pytest.raises(ValueError):
        oracle.rel_fro_slices(np.zeros((2, 1, 3)), np.zeros((2, 1, 4)), [(0, 2)])


def _mutant(fn, old, new):
    src = inspect.getsource(fn)
    assert src.count(old) == 1, (fn.__name__, old)
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    return ns[fn.__name__]


@pytest.mark.parametrize("old,new", [
    ("return float(num / den)", "return float(den / num)"),            # swapped
    ("return float(num / den)", "return float(num / den) ** 2"),       # squared norms
    ("num = np.linalg.norm((x - ref).ravel())",
     "num = np.abs(x - ref).sum()"),                                   # wrong norm
    ("den = np.linalg.norm(ref.ravel())", "den = np.linalg.norm(x.ravel())"),
    ("return float(num)", "return 0.0"),                               # zero reference
])
def test_rel_fro_mutants_fail(old, new):
    assert not _pins_rel_fro(_mutant(oracle.rel_fro, old, new))


@pytest.mark.parametrize("old,new", [
    ("rel_fro(x[s:e, h], ref[s:e, h])", "rel_fro(x[s:e], ref[s:e])"),        # heads pooled
    ("rel_fro(x[s:e, h], ref[s:e, h])", "rel_fro(x[s:e + 1, h], ref[s:e + 1, h])"),  # bound
    ("out[i, h] = ", "out[h % len(bounds), i % ref.shape[1]] = "),            # transposed
])
def test_rel_fro_slices_mutants_fail(old, new):
    assert not _pins_slices(_mutant(oracle.rel_fro_slices, old, new))

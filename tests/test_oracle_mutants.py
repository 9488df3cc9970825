"""The pins are strong enough: plausible mistakes planted in a copy of the oracle's C source
(compiled into a temporary library on the CPU) each fail at least one pin.

The committed oracle carries no mutation code; each mutant is a text substitution applied to
a temporary copy of ``oracle/recurrent.c``.
"""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "recurrent.c")

MUTANTS = {
    "decay dropped": ("S[i] *= alpha;", "S[i] *= 1.0;"),
    "decay sign": ("exp((double)a->g[row])", "exp(-(double)a->g[row])"),
    "update dropped": ("S[i * dv + j] += kd[i] * vd[j];", "S[i * dv + j] += 0.0 * kd[i];"),
    "update transposed": ("S[i * dv + j] += kd[i] * vd[j];",
                          "S[i * dv + j] += kd[j % dk] * vd[i % dv];"),
    "q and k swapped": ("qd[i] = widen_bf16(a->q[row * dk + i]);",
                        "qd[i] = widen_bf16(a->k[row * dk + i]);"),
    "gate index": ("exp((double)a->g[row])", "exp((double)a->g[t])"),
    "scale dropped": ("orow[j] = a->scale * acc;", "orow[j] = acc;"),
    "query reads transposed state": ("acc += qd[i] * S[i * dv + j];",
                                     "acc += qd[i] * S[(j * dk + i) % (dk * dv)];"),
    "h0 head/seq order": ("a->h0 + ((n * H + h) * dk) * dv", "a->h0 + ((h * a->nseq + n) * dk) * dv"),
    "first token skipped": ("for (int64_t t = bos; t < eos; ++t)",
                            "for (int64_t t = bos + (eos > bos); t < eos; ++t)"),
    "query before update": (
        "        /* step 2: add the outer product k^T v (row i of S gets k_i * v) */\n"
        "        for (int64_t i = 0; i < dk; ++i)\n"
        "            for (int64_t j = 0; j < dv; ++j)\n"
        "                S[i * dv + j] += kd[i] * vd[j];\n",
        ""),
}


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name!r} not found"
    if name == "query before update":
        # move the update after the query: drop it here, re-insert after the query block
        upd = old
        src = src.replace(upd, "")
        anchor = "    if (a->hT)\n"
        src = src.replace("        }\n    }\n" + anchor,
                          "        }\n" + upd + "    }\n" + anchor)
    else:
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", str(so),
                    str(path), "-lm"], check=True)
    return oracle.load_library(str(so))


def _pins_fail(lib) -> bool:
    """Run a few pins against ``lib``; True if any of them fails."""
    gen = torch.Generator().manual_seed(123)
    lens = [9, 0, 20]
    T, H, dk, dv = sum(lens), 2, 3, 5
    q = torch.randn((T, H, dk), generator=gen).to(torch.bfloat16)
    k = torch.randn((T, H, dk), generator=gen).to(torch.bfloat16)
    v = torch.randn((T, H, dv), generator=gen).to(torch.bfloat16)
    g = -torch.rand((T, H), generator=gen)
    h0 = torch.randn((len(lens), H, dk, dv), generator=gen)
    cu = torch.tensor([0, 9, 9, 29])
    o, hT = oracle.recurrent(q, k, v, g, 0.3, h0=h0, cu_seqlens=cu, _lib=lib)
    ob, hb = oracle.bruteforce(q, k, v, g, 0.3, h0=h0, cu_seqlens=cu)
    if not (oracle.rel_fro(o, ob) < 1e-12 and oracle.rel_fro(hT, hb) < 1e-12):
        return True
    # closed form with constant alpha
    a = 0.8
    gc = torch.full((T, H), math.log(a))
    _, hT = oracle.recurrent(q[:9], k[:9], v[:9], gc[:9], 1.0, h0=h0[:1],
                             cu_seqlens=torch.tensor([0, 9]), _lib=lib)
    kd, vd = k.double().numpy(), v.double().numpy()
    aa = math.exp(float(gc[0, 0]))
    for h in range(H):
        ref = aa ** 9 * h0[0, h].double().numpy()
        for i in range(1, 10):
            ref = ref + aa ** (9 - i) * np.outer(kd[i - 1, h], vd[i - 1, h])
        if not oracle.rel_fro(hT[0, h], ref) < 1e-12:
            return True
    return False


def test_committed_oracle_passes_the_pin_subset():
    assert not _pins_fail(oracle._load())


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, name, old, new)
    assert _pins_fail(lib), f"mutant {name!r} passed the pins"

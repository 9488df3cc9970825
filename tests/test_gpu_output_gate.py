"""Parity of the output norm and gate (sala_gla_output_norm_gate, through the C ABI) with the
fp64 oracle: relative Frobenius error <= 1e-2 over the whole output (bf16)."""
import numpy as np
import pytest
import torch

import oracle
from gated_linear_attention_gb300 import inputs

pytestmark = pytest.mark.gpu

O_TOL = 1e-2


@pytest.fixture(scope="module")
def sg():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from gated_linear_attention_gb300 import build, sala_gla
    build.build()
    return sala_gla


@pytest.mark.parametrize("T,H", [(1, 1), (5, 3), (37, 8), (41, 16), (300, 32), (19, 64), (20, 72)])
def test_output_gate_small(sg, T, H):
    x = inputs.make_output_gate(T, H, seed=T + H)
    out = sg.output_norm_gate(x["o"].cuda(), x["z"].cuda(), x["w"].cuda(), x["eps"])
    torch.cuda.synchronize()
    ref = oracle.output_norm_gate(x["o"], x["z"], x["w"], x["eps"]).reshape(T, H, 128)
    assert oracle.rel_fro(out.cpu().float(), ref) <= O_TOL


def test_output_gate_in_place_and_flat_layout(sg):
    x = inputs.make_output_gate(64, 32, seed=9)
    o = x["o"].cuda().reshape(64, 4096).contiguous()
    ref = sg.output_norm_gate(o, x["z"].cuda().reshape(64, 4096), x["w"].cuda(), x["eps"])
    sg.output_norm_gate(o, x["z"].cuda().reshape(64, 4096), x["w"].cuda(), x["eps"], out=o)
    torch.cuda.synchronize()
    assert torch.equal(o, ref)


def test_output_gate_full_size(sg):
    # the lightning layer's prefill shape (8192 tokens x 32 heads), every token checked
    x = inputs.make_output_gate()
    out = sg.output_norm_gate(x["o"].cuda(), x["z"].cuda(), x["w"].cuda(), x["eps"])
    torch.cuda.synchronize()
    ref = oracle.output_norm_gate(x["o"], x["z"], x["w"], x["eps"])
    assert oracle.rel_fro(out.cpu().float().reshape(ref.shape), ref) <= O_TOL
    # per-token errors stay small too (no token far off)
    err = np.linalg.norm(out.cpu().float().reshape(ref.shape).numpy() - ref, axis=1)
    assert np.max(err / np.linalg.norm(ref, axis=1)) <= 2e-2

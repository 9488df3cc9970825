"""Parity of the pooled decode step (sala_gla_recurrent_step_indexed, through the C ABI) with
the fp64 oracle: states gathered from and written back to a pool through slot indices, in
fp32 or bf16 storage.

Tolerances as for the plain decode: relative Frobenius error <= 1e-2 for o, <= 5e-3 for the
states. Padding rows, slots nobody names and out-of-range slots are checked exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from parity_report import record
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


def _run_steps(sg, x, pool, idx, steps):
    """`steps` pooled decode steps on the GPU; returns o [steps, N, H, 128] and the pool."""
    pd, idd = pool.cuda().clone(), idx.cuda()
    outs = []
    for s in range(steps):
        outs.append(sg.recurrent_step_indexed(x["q"][s].cuda(), x["k"][s].cuda(),
                                              x["v"][s].cuda(), x["g"][s].cuda(), x["scale"],
                                              pd, idd))
    torch.cuda.synchronize()
    assert sg.get_device_status() == 0
    return torch.stack(outs).cpu(), pd.cpu()


def _check_slices(o, o_ref, S, S_ref):
    """Worst (sequence, head) relative Frobenius errors of o [steps, N, H, d] over the steps,
    and of the states [N, H, d, d], within tolerance."""
    steps, N, H, d = o.shape
    of = o.float().transpose(0, 1).reshape(N * steps, H, d)
    orf = np.ascontiguousarray(np.asarray(o_ref).transpose(1, 0, 2, 3)).reshape(N * steps, H, d)
    so = oracle.rel_fro_slices(of, orf, [(n * steps, (n + 1) * steps) for n in range(N)])
    sh = oracle.rel_fro_slices(S.float(), S_ref, [(n, n + 1) for n in range(S.shape[0])])
    assert so.max() <= O_TOL, f"worst (sequence, head) output error {so.max():.3e}"
    assert sh.max() <= S_TOL, f"worst (sequence, head) state error {sh.max():.3e}"
    record({"o_slice_max": float(so.max()), "hT_slice_max": float(sh.max())})


def _ref_steps(x, pool, idx, steps, storage):
    ref = pool
    o_ref = []
    for s in range(steps):
        o, ref = oracle.recurrent_step_indexed(x["q"][s], x["k"][s], x["v"][s], x["g"][s],
                                               x["scale"], ref, idx, storage=storage)
        if storage == "bf16":
            ref = torch.from_numpy(ref).to(torch.bfloat16)   # exact: the values are bf16
        o_ref.append(o)
    return np.stack(o_ref), oracle._as_f64(ref)


@pytest.mark.parametrize("storage", ["f32", "bf16"])
@pytest.mark.parametrize("N,H,P,steps,pad", [(1, 1, 1, 1, ()), (6, 3, 10, 5, (1, 4)),
                                             (40, 32, 64, 3, (0, 39))])
def test_pool_decode_small(sg, storage, N, H, P, steps, pad):
    x = inputs.make_decode_steps("decode_pool", 0, steps, nseq=N, H=H)
    p = inputs.make_decode_pool(nseq=N, H=H, pool=P, storage=storage, pad=pad)
    o, pool = _run_steps(sg, x, p["pool"], p["indices"], steps)
    o_ref, pool_ref = _ref_steps(x, p["pool"], p["indices"], steps, storage)
    assert pool.dtype == p["pool"].dtype
    assert oracle.rel_fro(o.float(), o_ref) <= O_TOL
    named = [int(i) for i in p["indices"] if i >= 0]
    if named:
        assert oracle.rel_fro(pool[named].float(), pool_ref[named]) <= S_TOL
        live = [r for r in range(N) if int(p["indices"][r]) >= 0]
        _check_slices(o[:, live], o_ref[:, live], pool[p["indices"][live].long()],
                      pool_ref[p["indices"][live].long().numpy()])
    # padding rows give zeros; slots nobody names keep their bits
    for r in pad:
        assert torch.all(o[:, r] == 0)
    others = [i for i in range(P) if i not in named]
    assert torch.equal(pool[others], p["pool"][others])


def test_identity_indices_equal_dense_step(sg):
    # a pool addressed 0..N-1 in fp32 is the dense decode: bit-identical results
    N, H = 7, 4
    x = inputs.make_decode_steps("decode", 0, 2, nseq=N, H=H)
    S0 = inputs.make_decode_state("decode", nseq=N, H=H).cuda()
    S_dense, S_pool = S0.clone(), S0.clone()
    idx = torch.arange(N, dtype=torch.int32, device="cuda")
    for s in range(2):
        a = sg.recurrent_step(x["q"][s].cuda(), x["k"][s].cuda(), x["v"][s].cuda(),
                              x["g"][s].cuda(), x["scale"], S_dense)
        b = sg.recurrent_step_indexed(x["q"][s].cuda(), x["k"][s].cuda(), x["v"][s].cuda(),
                                      x["g"][s].cuda(), x["scale"], S_pool, idx)
        assert torch.equal(a, b)
    assert torch.equal(S_dense, S_pool)


def test_slot_past_the_pool_is_reported_and_skipped(sg):
    N, H, P = 3, 2, 4
    x = inputs.make_decode_steps("decode_pool", 0, 1, nseq=N, H=H)
    p = inputs.make_decode_pool(nseq=N, H=H, pool=P, storage="f32")
    idx = p["indices"].clone()
    idx[1] = P                                   # one past the end
    pool = p["pool"].cuda().clone()
    o = sg.recurrent_step_indexed(x["q"][0].cuda(), x["k"][0].cuda(), x["v"][0].cuda(),
                                  x["g"][0].cuda(), x["scale"], pool, idx.cuda())
    assert sg.get_device_status() == 8           # SALA_ERR_BAD_INDEX
    assert sg.get_device_status() == 0
    assert torch.all(o[1] == 0)
    untouched = [i for i in range(P) if i not in (int(idx[0]), int(idx[2]))]
    assert torch.equal(pool.cpu()[untouched], p["pool"][untouched])


def test_full_pool_decode_sampled_sequences(sg):
    # the benchmark's configuration (256 sequences, 32 heads, 512 bf16 slots), 100 steps;
    # four sequences checked against the oracle on a sub-pool of their slots
    w = inputs.WORKLOADS["decode_pool"]
    steps = 100
    x = inputs.make_decode_steps(w, 0, steps)
    p = inputs.make_decode_pool(w)
    o, pool = _run_steps(sg, x, p["pool"], p["indices"], steps)
    seqs = [0, 91, 170, 255]
    slots = p["indices"][seqs].long()
    xs = {n: x[n][:, seqs].contiguous() for n in ("q", "k", "v", "g")}
    xs["scale"] = x["scale"]
    o_ref, sub_ref = _ref_steps(xs, p["pool"][slots], torch.arange(len(seqs), dtype=torch.int32),
                                steps, "bf16")
    assert oracle.rel_fro(o[:, seqs].float(), o_ref) <= O_TOL
    assert oracle.rel_fro(pool[slots].float(), sub_ref) <= S_TOL
    _check_slices(o[:, seqs], o_ref, pool[slots], sub_ref)

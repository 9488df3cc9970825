"""The bench's multi-rank plumbing on CPU, world size 2 over gloo: the barrier and the max and
sum over ranks that its timing uses (the slowest rank's time; the units all ranks processed),
and the reference arm under torchrun, where rank 0 alone runs and prints one line and the
other rank exits 0 without work. (The data path itself has no collective: each rank runs its
own replica of the workload.) Last, on the oracle, the one exchange a split of a single
sequence by position over ranks would need: an all-gather of the segment summaries, after
which every rank's part equals the one-pass recurrence."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist()
    d.init("gloo")
    d.barrier()
    slowest = d.max(10.0 * rank + 1.5)     # per-rank elapsed time -> the job's time
    units = d.sum(100.0 * (rank + 1))      # per-rank work -> the job's work
    d.barrier()
    d.close()
    results.put((rank, slowest, units))


def test_dist_helper_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
    assert [p.exitcode for p in procs] == [0, 0]
    assert res == [(0, 11.5, 300.0), (1, 11.5, 300.0)]


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["value"] == line["value"] and line["cpu_baseline"]["kind"] == "oracle"


def _split_worker(rank, world, port, results):
    # One sequence split by position over the ranks: each rank summarises its segment as
    # (B_s, dS_s) = (sum of its g, its final state from a zero start), the summaries are
    # all-gathered, and each rank folds those of the ranks before it into its incoming state
    # (S_in(s+1) = exp(B_s) S_in(s) + dS_s) and runs its segment from there. The oracle does
    # the arithmetic; the exchange is the one collective such a split needs.
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist
    import oracle
    from gated_linear_attention_gb300 import inputs
    dist.init_process_group("gloo")
    x = inputs.make_prefill("varlen", seqlens=(192,), H=2, seed=3)
    T = 192
    a, b = rank * T // world, (rank + 1) * T // world
    sl = lambda t: t[a:b].contiguous()
    cu = torch.tensor([0, b - a], dtype=torch.int64)
    _, dS = oracle.recurrent(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), x["scale"], cu_seqlens=cu)
    B = sl(x["g"]).double().sum(0)                                   # [H]
    dS_all = [torch.zeros_like(torch.as_tensor(dS)) for _ in range(world)]
    B_all = [torch.zeros_like(B) for _ in range(world)]
    dist.all_gather(dS_all, torch.as_tensor(dS))
    dist.all_gather(B_all, B)
    S_in = x["h0"].double()
    for r in range(rank):
        S_in = torch.exp(B_all[r])[None, :, None, None] * S_in + dS_all[r]
    o, hT = oracle.recurrent(sl(x["q"]), sl(x["k"]), sl(x["v"]), sl(x["g"]), x["scale"],
                             h0=S_in, cu_seqlens=cu)
    o_full, h_full = oracle.recurrent(x["q"], x["k"], x["v"], x["g"], x["scale"], h0=x["h0"],
                                      cu_seqlens=torch.tensor([0, T], dtype=torch.int64))
    err_o = float(np.abs(np.asarray(o) - np.asarray(o_full)[a:b]).max() / np.abs(o_full).max())
    err_h = float(np.abs(np.asarray(hT) - np.asarray(h_full)).max() / np.abs(h_full).max())
    dist.destroy_process_group()
    results.put((rank, err_o, err_h if rank == world - 1 else 0.0))


def test_sequence_split_over_two_gloo_ranks_matches_one_pass():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_split_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, err_o, err_h in res:
        assert err_o <= 1e-12 and err_h <= 1e-12, (rank, err_o, err_h)

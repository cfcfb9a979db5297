"""The multi-rank host logic of bench.py on CPU ranks (gloo, world size 2).

Under torchrun every rank runs its own batch of the workload (weak scaling,
no data-path collective); the only collectives are the timing barrier and the
maximum of the per-rank times, taken here with the gloo backend.
"""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from workloads import WORKLOADS, make_scorer_inputs
    w = bench.rank_workload(WORKLOADS["topk_f32_t1024_k32"].with_(H=1, Tq=64, Tk=64), rank)
    q, _ = make_scorer_inputs(w)
    dist.barrier()
    mx = bench.max_over_ranks([rank + 1.0, 10.0 - rank, float(w.seed)], world, torch.device("cpu"))
    out[rank] = (mx, float(q.sum()), w.seed)
    dist.destroy_process_group()


def test_two_ranks_independent_batches_and_max_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    (mx0, s0, seed0), (mx1, s1, seed1) = res[0], res[1]
    assert mx0 == mx1 == [2.0, 10.0, float(max(seed0, seed1))]
    assert seed0 != seed1          # each rank its own batch
    assert s0 != s1                # ... so different inputs


def test_reference_arm_under_torchrun_prints_one_line():
    """bench.py --impl reference launched the way the multi-GPU runs launch it
    (torchrun, two ranks): rank 0 alone runs the oracle and prints one JSON
    line, the other rank exits 0 without work."""
    import json
    import subprocess
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3", "--workload", "topk_f32_t1024_k32", "--cpu-rows", "128"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0

"""Host-side multi-rank logic of bench.py on CPU with gloo (world size 2).

Each rank runs an independent replica (other seeds, same shapes); the job's
time is the max over ranks; the reference arm runs on rank 0 only."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from top_sparse_attention_exact_gb300 import synth
    w = synth.WORKLOADS["qwen7b_16k"]
    wr = bench.replica_workload(w, rank)
    tot = bench.max_over_ranks(10.0 * (rank + 1), dist, "cpu")
    dist.barrier()
    q.put((rank, wr.seeds, (wr.B, wr.Hq, wr.Hkv, wr.L0), tot))
    dist.destroy_process_group()


def test_replicas_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, sh0, t0), (r1, s1, sh1, t1) = res
    assert set(s0).isdisjoint(s1)            # independent replicas
    assert sh0 == sh1                        # same per-rank work (weak scaling)
    assert t0 == t1 == 20.0                  # the slowest rank's time


def _bench_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--workload", "tiny_1h_2k", "--steps", "3", "--warmup", "1"],
                          capture_output=True, text=True, env=env, timeout=600)


def test_reference_arm_runs_on_rank0_only():
    r1 = _bench_reference(1, 2)
    assert r1.returncode == 0, r1.stderr
    assert r1.stdout.strip() == ""
    r0 = _bench_reference(0, 1)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "us/step/layer"
    assert line["higher_is_better"] is False and line["steps"] == 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0

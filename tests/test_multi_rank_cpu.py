"""The replica (N > 1) host logic of bench.py on two gloo ranks, CPU only.

The block's data-parallel path has no exchange step, so N GPUs run N
independent replicas; what the job reports is every rank's tokens over the
slowest rank's time. These checks run that aggregation across real
processes, plus the per-rank inputs and the reference arm's rank-0-only output.
"""
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


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    from llama_family_decoder_gb300.synth import WORKLOADS, make_input
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    local_ms = [120.0, 150.0][rank]  # rank 1 is the slow one
    total = bench.max_over_ranks(local_ms, "cpu")
    value = bench.job_tokens_per_s(world, 2048, 10, total)
    wl = WORKLOADS["tiny_f32_T64_D256"]
    x = make_input(wl, seed=bench.rank_seed(wl, rank))
    dist.barrier()
    dist.destroy_process_group()
    out.put((rank, total, value, float(x.sum())))


def test_two_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, v0, s0), (r1, t1, v1, s1) = res
    assert t0 == t1 == 150.0  # both ranks see the job's (slowest) time
    assert v0 == v1 == 2 * 2048 * 10 / 0.150
    assert s0 != s1  # each replica decodes its own synthetic batch


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                        "--warmup", "0", "--workload", "tiny_f32_T64_D256"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""

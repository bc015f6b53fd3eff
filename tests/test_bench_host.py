"""Host logic of bench.py without a GPU: the replicas path across two gloo ranks (barrier,
max over ranks, rank-0-only reference arm) and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    # each rank's own step time; the job's time is the slowest rank's
    t = bench.max_over_ranks(10.0 + rank, world)

    class Args:
        workload = bench.VerifyLogitsWorkload.name
        warmup, steps, gpus = 1, 1, world
    skipped = rank != 0 and bench.run_reference(Args) is None
    out.put((rank, t, skipped))
    bench.barrier(world)
    dist.destroy_process_group()


def test_replicas_two_gloo_ranks():
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
    assert [r[1] for r in res] == [11.0, 11.0]       # max over ranks on every rank
    assert res[1][2]                                  # rank 1 runs no reference arm


def test_reference_arm_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "verify-logits-b64-k4",
                        "--steps", "1", "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["higher_is_better"] is True
    assert line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "verify-logits-b64-k4"


def test_workloads_registered():
    sys.path.insert(0, ROOT)
    import bench
    assert set(bench.WORKLOADS) == {"dense-8b-verify-k4", "verify-logits-b64-k4", "serving-8b-b32-k8",
                                    "sampling-27b-0p8b"}


def test_dense_oracle_step_is_one_whole_verify_step():
    """The CPU baseline and the reference arm time the same oracle step: K + 1 tokens through
    every layer plus the lm_head, counted at the scripted drafter's closed-form mean."""
    sys.path.insert(0, ROOT)
    import bench
    import synth
    step, sample = bench.dense_oracle_step(synth.SMALL_BF16, 4, 0.7)
    assert abs(step() - (1 - 0.7 ** 5) / 0.3) < 1e-12
    assert "through 2 layers" in sample and "4096-row lm_head" in sample

"""The multi-rank bench path on CPU: two gloo ranks, the max-over-ranks timing reduction and the
weak-scaling aggregate (replicas: each rank runs its own requests; no data-path collective)."""
import os
import socket
import sys

import pytest
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r measured (1 + r) ms per step and (3 - r) ms end to end: every rank must see the max of each
    got = bench.max_over_ranks([1.0 + rank, 3.0 - rank], "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1] == [2.0, 3.0]


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], "cpu") == [1.5, 2.5]


def test_weak_scaling_aggregate_and_config():
    sys.path.insert(0, ROOT)
    import bench
    from compressed_sparse_attention_c4a_gb300 import synth
    spec = synth.case_specs()["c4a_decode_batch"]
    # whole-job throughput: every rank serves its own 32 requests in the (max) step time
    assert bench.queries_per_step(spec) == 32
    assert bench.algorithmic_bytes(spec) == (69201792, 20971520)
    cfg = bench.workload_config("c4a_decode_batch", spec, 4)
    assert cfg["parallelism"] == "replicas x4" and cfg["batch"] == 32


def test_gpus_flag_starts_that_many_ranks():
    """``bench.py --gpus 2`` outside a launcher starts two ranks itself (torch.distributed.run on 127.0.0.1);
    rank 0 prints the one JSON line with n_gpus = 2, the other rank exits without work (the oracle arm, so
    this runs on CPU)."""
    import json
    import subprocess
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                          "--workload", "c4a_tiny_decode", "--steps", "1", "--warmup", "0", "--cpu-seconds", "0.5"],
                         capture_output=True, text=True, timeout=600, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["config"]["parallelism"] == "replicas x2"


def test_gpus_flag_inside_a_launcher_must_match_world_size():
    import subprocess
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                          "--workload", "c4a_tiny_decode", "--steps", "1"], capture_output=True, text=True, timeout=300,
                         env=env)
    assert res.returncode != 0 and "launcher of 1 rank" in res.stderr

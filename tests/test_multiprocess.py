"""The multi-process paths of bench.py on CPU (no GPU): the path shards by
sequence into independent replicas, so the only exchange is the timing
reduction -- every rank ends with the maximum over ranks -- and under a
multi-rank launch the reference arm runs on rank 0 alone (other ranks exit 0
and print nothing). Two gloo ranks on 127.0.0.1."""
import json
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 7.5 * rank           # each rank's own timing
        got = bench.max_over_ranks(mine, dist)
        alone = bench.max_over_ranks(mine, None)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"mine": mine, "got": got, "alone": alone}, f)
    finally:
        dist.destroy_process_group()


def test_timing_reduction_is_the_max_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    mp.start_processes(_rank, args=(world, port, str(tmp_path)), nprocs=world, join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    top = max(r["mine"] for r in res)
    for r in res:
        assert r["got"] == top            # every rank holds the maximum
        assert r["alone"] == r["mine"]    # no process group: the value itself


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3", "--gpus", "2"], capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)
    assert r.returncode == 0
    assert r.stdout.strip() == ""

"""The N > 1 host logic of bench.py on CPU: two ranks over gloo (127.0.0.1),
each with its own timing; both must agree on the slowest rank's time, the
whole-job throughput must count every rank's units, the rank/world
environment must be read as torchrun sets it, and the reference arm must
leave ranks other than 0 without work."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    env = bench.dist_env()
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # per-rank timings: rank 1 is slower on the first, rank 0 on the second
        mine = [10.0 + 5.0 * rank, 7.0 - 2.0 * rank]
        merged = bench.max_over_ranks(mine, "cpu", world)
        dist.barrier()
        value = bench.job_throughput(32 * 50, world, merged[0])

        class Args:
            workload, steps, warmup = None, 1, 0
        ref = bench.run_reference(Args(), rank, world, rank) if rank != 0 else "skipped on rank 0"
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"env": env, "mine": mine, "merged": merged, "value": value, "ref": ref}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["env"] == [r, world, r]
        assert d["merged"] == [15.0, 7.0]            # element-wise max over the ranks
        assert d["value"] == pytest.approx(32 * 50 * world / 15e-3)
    assert res[1]["ref"] is None                     # the reference arm runs on rank 0 only


def test_single_rank_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5], "cpu", 1) == [3.0, 4.5]
    assert bench.job_throughput(100, 1, 1000.0) == pytest.approx(100.0)

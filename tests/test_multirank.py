"""The N > 1 path of bench.py on CPU with two gloo ranks: the max-over-ranks timing reduction, the barrier,
and the reference arm running on rank 0 only.  (Every rank runs an independent problem; there is no
collective on the data path, only this timing reduction.)"""
import json
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    bench.init_dist(world, "gloo")
    local_ms = 1.0 + rank * 2.5
    got = bench.max_over_ranks(local_ms, world)
    bench.barrier(world)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": got, "env": list(bench.dist_env())}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_time(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [r["max"] for r in res] == [3.5, 3.5]
    assert [r["env"] for r in res] == [[2, 0, 0], [2, 1, 1]]


def test_reference_arm_prints_nothing_on_other_ranks(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    assert capsys.readouterr().out == ""

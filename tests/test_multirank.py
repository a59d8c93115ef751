"""Host-side multi-rank logic of the benchmark, on CPU with gloo (world size 2).

Decode shards by sequence: every rank runs an independent replica with its
own seeds (weak scaling, no collective on the data path).  The only
collectives are the barrier around the timed region and the max over ranks
of the measured time."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as tmp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    got_rank, got_world = bench.init_ranks("gloo")
    assert (got_rank, got_world) == (rank, world)
    bench.barrier()
    local_ms = 10.0 + 5.0 * rank
    out[rank] = (bench.max_over_ranks(local_ms), bench.rank_seed(0, rank))
    bench.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_max_time_and_distinct_seeds():
    world = 2
    port = _free_port()
    manager = tmp.get_context("spawn").Manager()
    out = manager.dict()
    tmp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] != out[1][1]


def test_single_rank_is_identity(monkeypatch):
    for var in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(var, raising=False)
    assert bench.rank_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_ranks_other_than_zero_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.run_reference(bench.parse_args(["--impl", "reference"])) == 0

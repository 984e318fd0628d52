"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1), each timing
its own replica; the job's time is the maximum over ranks on every rank, and
a non-zero rank of the reference arm does no work and prints nothing."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b = _bench()
    assert b._dist() == (world, rank, rank)
    mine = 1.0 + 0.5 * rank                  # each replica's own step time (ms)
    got = b._max_over_ranks(mine, torch.device("cpu"), world)
    dist.barrier()
    dist.destroy_process_group()
    out[rank] = got


def test_two_gloo_ranks_take_the_max():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True,
                       start_method="spawn")
    assert dict(out) == {0: 1.5, 1: 1.5}


def test_single_rank_keeps_its_value():
    assert _bench()._max_over_ranks(2.25, torch.device("cpu"), 1) == 2.25


def test_reference_arm_other_ranks_do_nothing(capsys, monkeypatch):
    b = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert b.run_reference(None, None) is None   # returns before touching args or cfg
    assert capsys.readouterr().out == ""

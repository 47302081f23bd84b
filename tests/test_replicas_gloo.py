"""The multi-process path of bench.py on the CPU: two gloo ranks run the
replica set-up, barrier and max-over-ranks timing that `bench.py --gpus N`
uses under torchrun.  No data-path collective exists ("replicas only")."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # Each rank reports a different elapsed time; every rank must see the max.
    got = bench.max_over_ranks(10.0 + rank, w)
    out[rank] = got
    dist.destroy_process_group()


def test_two_rank_replica_timing():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert dict(out) == {0: 11.0, 1: 11.0}


def test_reference_arm_other_ranks_exit_quietly(capsys, monkeypatch):
    """Under torchrun only rank 0 runs and prints the reference arm."""
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        ref_rows, steps, warmup = 4, 1, 0

    from context_ring_attention_cpattn_gb300.workloads import WORKLOADS

    assert bench.run_reference(Args, WORKLOADS["tiny"]) == 0
    assert capsys.readouterr().out == ""

"""The multi-process path of bench.py on CPU: two gloo ranks on 127.0.0.1 (no GPU).

Each rank runs its own replica of the stack on its own seeded layers (weak scaling, no
data-path collective); the ranks only meet for a barrier and the max of their times.
These tests check that host logic: process-group setup, the barrier, the max over
ranks, that the ranks' synthetic layers are distinct, the whole-job throughput, and that
only rank 0 of the reference arm does any work."""
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + rank, w)
    ids = bench.rank_layer_ids(rank, 32)
    # a rank's time and the job value computed from the max over ranks
    v = bench.job_value(1000, m, w)

    class A:
        steps, warmup, gpus = 1, 0, world

    rc = bench.run_reference(A()) if rank != 0 else None
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": m, "ids": ids, "value": v, "ref_rc": rc}, f)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path, capfd):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    # every rank sees the slowest rank's time
    assert [r["max"] for r in res] == [11.0, 11.0]
    # the ranks' layers are distinct
    assert not set(res[0]["ids"]) & set(res[1]["ids"])
    assert len(set(res[0]["ids"])) == 32
    # whole-job throughput: all ranks' entries over the max time
    assert res[0]["value"] == pytest.approx(2 * 1000 / 11.0e-3)
    # the reference arm on a rank other than 0 returns 0 and prints nothing
    assert res[1]["ref_rc"] == 0
    assert "reference" not in capfd.readouterr().out


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.rank_layer_ids(0, 3) == [0, 1, 2]
    assert bench.job_value(500, 2.0, 1) == pytest.approx(250000.0)

"""The N > 1 path of bench.py on CPU: two ranks over gloo (127.0.0.1), through
the same helpers the GPU run uses under torchrun. Each rank runs the step on
its own tokens (weak scaling; the weight-gradient all-reduce of data
parallelism is tested in test_dp_cpu.py); the timed region ends with a barrier
and the slowest rank's time, taken with an all-reduce MAX, is what every rank
reports."""
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    r, local, w = bench.dist_init()
    assert (r, local, w) == (rank, rank, world)
    # each rank "times" a different amount of work; everyone reports the max
    t = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    bench.barrier(w)
    seed = bench.rank_seed(r)
    import torch.distributed as dist
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "max_ms": t, "seed": seed}, f)


def test_two_ranks_gloo_max_over_ranks(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert [x["max_ms"] for x in res] == [15.0, 15.0]       # the slowest rank's time
    assert len({x["seed"] for x in res}) == world           # each rank its own tokens
    assert all(x["world"] == world for x in res)


def test_single_process_needs_no_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    assert bench.dist_init() == (0, 0, 1)
    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)


def test_reference_arm_runs_on_rank0_only(capsys):
    """Under torchrun the reference arm (the fp64 oracle on the host cores)
    runs and prints on rank 0 alone; the other ranks return without work."""
    import argparse
    import time
    import bench
    args = argparse.Namespace(workload="1b-T16384-d2048-r512-dff5461", steps=3, warmup=3)
    t0 = time.perf_counter()
    bench.run_reference(args, rank=1, world=2)
    assert time.perf_counter() - t0 < 1.0
    assert capsys.readouterr().out == ""


def test_gpus_flag_must_match_the_launch(monkeypatch):
    """--gpus N without N launched processes is an error, not a silent 1-GPU run."""
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    import bench
    with pytest.raises(SystemExit) as e:
        bench.main(["--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert "--gpus 2" in str(e.value)

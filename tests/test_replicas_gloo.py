"""Multi-GPU runs are independent replicas (routing is token-local, so nothing
is exchanged on the data path): the benchmark's host logic across ranks is the
per-rank seeding of the inputs, the max-over-ranks step time and the whole-job
rate. Checked here with two gloo ranks on the CPU."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import synthetic

    assert bench.dist_env() == (rank, world, rank)
    # every rank times its own replica; the job's time is the slowest rank's
    slowest = bench.reduce_max(1.5 + rank, "cpu")
    shape, recipe, _ = synthetic.decode_layer(8)
    x, logits = bench.host_inputs(shape, recipe, 2, rank)
    np.save(os.path.join(out_dir, f"x{rank}.npy"), x)
    np.save(os.path.join(out_dir, f"logits{rank}.npy"), logits)
    with open(os.path.join(out_dir, f"max{rank}.txt"), "w") as f:
        f.write(repr(slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    for r in range(world):
        assert float(open(tmp_path / f"max{r}.txt").read()) == 2.5
    # replicas draw different tokens and router logits (independent problems)
    assert not np.array_equal(np.load(tmp_path / "x0.npy"), np.load(tmp_path / "x1.npy"))
    assert not np.array_equal(np.load(tmp_path / "logits0.npy"), np.load(tmp_path / "logits1.npy"))


def test_job_rate_and_single_rank():
    import bench

    # 8 tokens x 48 layers per rank, 2 ranks, 2.5 ms for the slowest rank
    assert bench.job_rate(8 * 48, 2, 2.5e-3) == pytest.approx(307200.0)
    # without a process group the step time is the rank's own
    assert bench.reduce_max(3.25, "cpu") == 3.25

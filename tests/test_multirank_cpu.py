"""The benchmark's multi-rank logic on CPU: two gloo ranks, as torchrun would
launch them.  The convolution shards over the batch with no exchange step,
so the only cross-rank operation is the max-over-ranks of the elapsed time;
the reference arm runs on rank 0 alone."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.init_dist(w, "gloo")
    got = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    bench.barrier(w)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)


def _ref_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import io
    import contextlib
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        # only rank 0 does the work; the other rank must return at once
        if rank == 1:
            bench.run_reference(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"]))
    out[rank] = buf.getvalue()


def test_reference_arm_other_ranks_exit_without_work():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_ref_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[1] == ""

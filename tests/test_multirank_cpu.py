"""The N > 1 path of bench.py on the CPU: two gloo ranks, independent batches,
max-over-ranks timing and the whole-job value (no GPU, no collective on the
data path)."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workloads import config_workload


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = config_workload(1, seed=bench.rank_seed(20261, rank))
    fake_ms = [1.0 + rank, 10.0 - rank, 5.0]
    bench._barrier(dist)
    mx = bench._max_ranks(fake_ms, dist, torch, device="cpu")
    digest = torch.tensor([int(wl.q[:64].astype(np.int64).sum())], dtype=torch.int64)
    gathered = [torch.zeros_like(digest) for _ in range(world)]
    dist.all_gather(gathered, digest)
    out[rank] = (mx, [int(g.item()) for g in gathered])
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == [2.0, 10.0, 5.0]  # max over ranks, element-wise
    d0, d1 = res[0][1]
    assert d0 != d1  # each rank drew its own batch
    assert bench.whole_job_value(100.0, world, 2.0) == 100.0


class _FakeLibraryBuild:
    """Stands in for the package's build step: 'compiles' (slowly, leaving a marker) only when
    the marker is missing, and counts its compiles in a file, one line per compile."""

    def __init__(self, root):
        self.marker = os.path.join(root, "libpkv.so")
        self.log = os.path.join(root, "compiles.txt")

    def library_is_fresh(self):
        return os.path.exists(self.marker)

    def build(self):
        if self.library_is_fresh():
            return
        import time

        time.sleep(0.5)  # long enough that an unsynchronised second rank would also start compiling
        with open(self.log, "a") as f:
            f.write(f"{os.getpid()}\n")
        with open(self.marker, "w") as f:
            f.write("built")


def _build_worker(rank, world, port, root):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.build_library(_FakeLibraryBuild(root), dist, local_rank=rank)
    dist.destroy_process_group()


def test_ranks_of_a_node_compile_once(tmp_path):
    world = 2
    mp.spawn(_build_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    with open(tmp_path / "compiles.txt") as f:
        assert len(f.read().split()) == 1  # local rank 0 compiled; rank 1 waited and found it fresh


def test_single_rank_is_identity():
    assert bench._max_ranks([1.0, 2.0], None, torch) == [1.0, 2.0]
    assert bench.rank_seed(5, 0) == 5

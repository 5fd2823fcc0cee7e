"""The N > 1 path of bench.py on CPU: two ranks over gloo (127.0.0.1).

bench.py runs one independent replica of the workload per rank ("replicas
only": the grouped GEMM has no exchange step), brackets the timed steps
with barriers and reports the maximum step time over ranks. Here two
processes run its rank set-up, barrier and max-over-ranks reduction with
gloo, without a GPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    mx = bench.max_over_ranks(w, 10.0 + 3.0 * rank, "cpu")
    bench.barrier(w)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(repr(mx))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_step_time(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(world)]
    assert got == [13.0, 13.0]

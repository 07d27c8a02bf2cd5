"""The multi-rank path of bench.py on CPU: two gloo ranks set up from the
launcher's environment, meet at the barrier and agree on the maximum of their
timings (the bench reports the slowest rank's time for the whole job)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    # the ranks run on the CPU even where a GPU is present (gloo)
    os.environ.update({"CUDA_VISIBLE_DEVICES": "", "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup()
    bench.barrier(w)
    m = bench.max_over_ranks(1.5 + r, w)
    with open(os.path.join(out_dir, f"rank{r}.txt"), "w") as f:
        f.write(f"{r} {w} {local} {m} {dist.get_backend()}\n")
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_max(tmp_path):
    pytest.importorskip("torch")
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, str(tmp_path))) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        rr, ww, local, m, backend = open(tmp_path / f"rank{r}.txt").read().split()
        assert (int(rr), int(ww), int(local)) == (r, world, r)
        assert float(m) == 2.5
        assert backend == "gloo"

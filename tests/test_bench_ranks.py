"""The bench's multi-process path on CPU: two gloo ranks (one process each,
as torchrun launches them) set up the process group the way bench.py does,
meet at its barrier and agree on the max-over-ranks time that the whole-job
throughput divides by.  The decode path has no data-path collective (each
rank is an independent replica), so this is the only cross-rank code."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, local, w = bench.dist_setup(world)
    assert (r, local, w) == (rank, rank, world) and dist.get_backend() == "gloo"
    bench.barrier(w)
    elapsed_ms = 10.0 + 5.0 * rank            # each rank's own timed region
    out[rank] = bench.max_over_ranks(elapsed_ms, w)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        result = dict(out)
    assert codes == [0, 0], codes
    # every rank reports the slowest rank's time: whole-job tokens / that time
    assert result == {0: 15.0, 1: 15.0}


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    if "WORLD_SIZE" in os.environ:
        pytest.skip("running under a launcher")
    assert bench.dist_setup(1) == (0, 0, 1)
    assert bench.max_over_ranks(3.5, 1) == 3.5

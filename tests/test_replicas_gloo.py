"""The multi-process host logic of bench.py on CPU: two ranks over gloo.

The path runs replicas only (sequences never exchange data), so the cross-rank
pieces are the timing barrier, the max-over-ranks reduction of the timed
durations, the aggregate over all ranks' tokens, and rank 0 alone printing the
reference arm. Each rank runs in its own spawned process; the rendezvous is on
127.0.0.1.
"""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, _ = bench.dist_env()
    # per-rank timings (ms): the job time is the slowest rank's
    local = [10.0 + 2.0 * rank, 3.0 - rank]
    got = bench.reduce_max(local, w)
    bench.barrier(w)
    # the reference arm: rank 0 alone runs the oracle sample and prints its line
    buf = io.StringIO()
    args = type("A", (), {"steps": 1, "warmup": 0})()
    if r != 0:
        with redirect_stdout(buf):
            bench.run_reference(args)
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "max": got, "ref_out": buf.getvalue()}, f)


def test_two_ranks_reduce_max_barrier_and_rank0_only_reference(tmp_path):
    import torch.multiprocessing as mp
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["world"] == world and d["rank"] == r
        assert d["max"] == [12.0, 3.0]   # element-wise max over the ranks' values
    assert res[1]["ref_out"] == ""       # a rank other than 0 does no work and prints nothing


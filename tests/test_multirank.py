"""The multi-rank path on the CPU (gloo, world size 2).

Sequences are independent, so N ranks each take their own shard of
sequences and share nothing on the data path; only the timing is combined
(the job ends when the slowest rank does) and the work is summed. These
tests run that host-side logic in two gloo processes."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, name, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        wl = bench.rank_workload(name, rank)
        run = oracle.run(wl, decode=False)            # this rank's own pool and cache
        my_time = 1.0 + 0.5 * rank                     # stand-in for the rank's step time
        t_max = bench.max_over_ranks(my_time, world)
        job_bytes = bench.sum_over_ranks(float(bench.step_bytes(wl)["step"]), world)
        job_seqs = bench.sum_over_ranks(float(wl.num_seqs), world)
        out.put((rank, t_max, job_bytes, job_seqs, list(wl.context_lens),
                 float(wl.q.float().sum()), run.pool.stats(), bench.step_bytes(wl)["step"]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["tiny", "llama3_8b"])
def test_two_ranks_take_disjoint_shards_and_combine_timing(name):
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, name, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, t0, b0, s0, lens0, q0, st0, mine0), (_, t1, b1, s1, lens1, q1, st1, mine1) = res
    assert t0 == t1 == 1.5                     # both ranks report the slowest rank's time
    assert b0 == b1 == mine0 + mine1           # the job's bytes are both shards'
    assert s0 == s1
    assert q0 != q1                            # different sequences (values) per rank
    if name == "llama3_8b":
        assert lens0 != lens1                  # and different lengths

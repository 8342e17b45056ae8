"""The multi-rank path of bench.py on CPU: two gloo ranks, each with its own
timings; the job rate is both ranks' units over the slower rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [0.5 + rank, 2.0 - rank]                 # rank 1 is slower on the first
    worst = bench.slowest(mine)
    rate = bench.whole_job_rate(1000.0, worst[0], world)
    q.put((rank, worst, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, rate in out:
        assert worst == [1.5, 2.0]
        assert rate == pytest.approx(2000.0 / 1.5)


def test_single_process_keeps_its_timings():
    import bench
    assert bench.slowest([1.0, 2.0]) == [1.0, 2.0]
    assert bench.whole_job_rate(10.0, 2.0, 1) == 5.0


def test_percentiles_nearest_rank():
    import bench
    assert bench.percentiles([]) is None
    assert bench.percentiles([3.0]) == {"p10": 3.0, "p50": 3.0, "p90": 3.0}
    got = bench.percentiles([float(x) for x in range(10, 0, -1)])   # 10 .. 1, unsorted
    assert got == {"p10": 2.0, "p50": 5.0, "p90": 9.0}


def test_num_seqs_option_shrinks_the_batch():
    import bench
    from paged_kv_cache_130_gb300 import workloads as W
    args = bench.parse_args(["--workload", "opt13b_f16", "--num-seqs", "4"])
    assert args.num_seqs == 4
    w = W.make(args.workload, num_seqs=args.num_seqs)
    assert w.num_seqs == 4 and w.q.shape[0] == 4 and w.block_tables.shape[0] == 4
    assert W.make(args.workload).num_seqs == 32
    assert bench.parse_args([]).num_seqs is None

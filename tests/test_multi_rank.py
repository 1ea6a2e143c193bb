"""The multi-rank path of bench.py on CPU: two gloo ranks, each holding its
own replica of a workload (the decode units are independent, so several
GPUs run replicas with no collective on the data path).  What the ranks do
share is checked here: the elapsed time is the maximum over ranks, the job
value counts every rank's bytes, replicas are seeded apart, and the
reference arm runs on rank 0 only."""
import argparse
import os
import socket

import torch
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist

    import oracle
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        w = workloads.make_workload(1, seed=bench.replica_seed(1, rank))
        flat = w.pool.view(-1)
        out, err = oracle.attention_decode(w.q, flat, flat[w.v_offset:], w.block_table, w.lens,
                                           w.scale, num_kv_heads=w.Hkv, block_size=w.bs,
                                           block_stride=w.block_stride, num_blocks=w.NB)
        mine = torch.tensor([float(out.sum())], dtype=torch.float64)
        every = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(every, mine)
        results.put((rank, elapsed, int(err.any()), [float(x) for x in every]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_only_the_clock():
    ctx = mp.get_context("spawn")
    results = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(results.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, e0, all0), (r1, t1, e1, all1) = got
    assert (r0, r1) == (0, 1)
    assert t0 == t1 == 15.0                      # the slowest rank's time on every rank
    assert e0 == e1 == 0
    assert all0 == all1 and all0[0] != all0[1]   # independent replicas
    assert bench.replica_seed(1, 0) != bench.replica_seed(1, 1)


def test_job_value_counts_every_rank():
    assert bench.job_throughput(1, 2_000_000_000, 1.0) == 2000.0
    assert bench.job_throughput(4, 2_000_000_000, 1.0) == 8000.0
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(workload=1, block_size=None, batch=None, long_seq=0, int8=False,
                              steps=2, warmup=1)
    bench.run_reference(args)
    assert capsys.readouterr().out == ""

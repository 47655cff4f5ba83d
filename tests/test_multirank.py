"""The N > 1 host path of bench.py on CPU: two gloo ranks, each with its own independent
group, combine their timings (max) and their work (sum) without any data-path collective."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 1000.0 + 250.0 * rank               # rank 1 is the slow one
    flops = 1e15 * (rank + 1)
    out[rank] = (bench.rank_max(ms, dist), bench.rank_sum(flops, dist))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_time_and_work():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        mx, sm = res[rank]
        assert mx == 1250.0
        assert sm == 3e15
    # whole-job throughput = all ranks' work / the slowest rank's time
    assert res[0][1] / (res[0][0] / 1e3) == pytest.approx(2.4e15)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--workload", "tiny"])
    bench.main()
    assert capsys.readouterr().out == ""

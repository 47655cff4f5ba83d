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


def _cp_worker(rank, world, port, out):
    """One rank of a context-parallel replay on CPU: its partial attention over its prompt
    shard (float64 oracle standing in for the shard kernel), the library's all-gather of
    the partials, the oracle merge; then its dq part and the library's fp32 reduction."""
    import numpy as np
    import torch.distributed as dist
    import oracle
    from long_context_grpo_gb300 import cp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(0)                 # same draw on every rank
    P, T, D = 37, 5, 16
    q = rng.normal(size=(T, D))
    k = rng.normal(size=(P, D))
    v = rng.normal(size=(P, D))
    b = cp.shard_bounds(P, world)
    s = q @ k[b[rank]:b[rank + 1]].T / np.sqrt(D)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    o_r = torch.tensor(e @ v[b[rank]:b[rank + 1]] / e.sum(axis=1, keepdims=True))
    lse_r = torch.tensor(m[:, 0] + np.log(e.sum(axis=1)))
    o_all, lse_all = cp.exchange_partials(o_r, lse_r)
    o, lse = oracle.merge_partials([x.numpy() for x in o_all], [x.numpy() for x in lse_all])
    dq = cp.reduce_dq(torch.full((T, D), float(rank + 1), dtype=torch.bfloat16))
    out[rank] = (o, lse, dq.float().numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_context_parallel_exchange_on_two_gloo_ranks():
    import numpy as np
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_cp_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    rng = np.random.default_rng(0)
    P, T, D = 37, 5, 16
    q = rng.normal(size=(T, D))
    k = rng.normal(size=(P, D))
    v = rng.normal(size=(P, D))
    s = q @ k.T / np.sqrt(D)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    o_ref = e @ v / e.sum(axis=1, keepdims=True)
    lse_ref = m[:, 0] + np.log(e.sum(axis=1))
    for rank in (0, 1):
        o, lse, dq = res[rank]
        assert np.allclose(o, o_ref, atol=1e-12) and np.allclose(lse, lse_ref, atol=1e-12)
        assert np.all(dq == 3.0)                    # 1 + 2 summed over the two ranks


def test_shard_bounds_cover_the_prompt_once():
    from long_context_grpo_gb300 import cp
    for P, world in ((37, 2), (2097152, 8), (8, 8), (1000, 3)):
        b = cp.shard_bounds(P, world)
        assert b[0] == 0 and b[-1] == P and len(b) == world + 1
        sizes = [y - x for x, y in zip(b[:-1], b[1:])]
        assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        cp.shard_bounds(3, 4)

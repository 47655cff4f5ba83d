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


class _HostOps:
    """Test stand-in for the library's merge and conversions (float64 CPU tensors)."""

    @staticmethod
    def merge(o_parts, lse_parts):
        import oracle
        o, lse = oracle.merge_partials([x.numpy() for x in o_parts], [x.numpy() for x in lse_parts])
        return torch.tensor(o), torch.tensor(lse)

    @staticmethod
    def to_f32(x):
        return x.clone()

    @staticmethod
    def to_bf16(x):
        return x.clone()


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
    dq = cp.reduce_dq(torch.full((T, D), float(rank + 1), dtype=torch.bfloat16), ops=_BfOps)
    out[rank] = (o, lse, dq.float().numpy())
    dist.barrier()
    dist.destroy_process_group()


class _BfOps:
    """bf16 <-> fp32 conversions as torch does them (CPU stand-in for the library's)."""

    @staticmethod
    def to_f32(x):
        return x.to(torch.float32)

    @staticmethod
    def to_bf16(x):
        return x.to(torch.bfloat16)


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


# ---------------------------------------------------------------- cp.replay_response itself
_CP_CASE = dict(P=29, R=6, D=8, seed=11)


def _cp_inputs():
    import numpy as np
    c = _CP_CASE
    rng = np.random.default_rng(c["seed"])
    mk = lambda *shape: torch.tensor(rng.normal(size=shape) * 0.7)   # noqa: E731
    kp, vp = mk(c["P"], 1, c["D"]), mk(c["P"], 1, c["D"])
    q, ks, vs = mk(c["R"], 1, c["D"]), mk(c["R"], 1, c["D"]), mk(c["R"], 1, c["D"])
    do = torch.tensor(rng.normal(size=(c["R"], 1, c["D"])))
    return kp, vp, q, ks, vs, do


class _ShardStandIn:
    """Test stand-in for a Prefix over one prompt shard (one head, float64 on the CPU): the
    partial attention of the queries over the shard's keys (and, for the suffix owner, the
    causal suffix), and the shard backward with the merged o and lse.  Records which calls
    the rank made and keeps its prompt-key gradients."""

    def __init__(self, kp, vp):
        self.kp, self.vp = kp[:, 0], vp[:, 0]
        self.s = 1.0 / float(kp.shape[-1]) ** 0.5
        self.calls = []
        self.dk = torch.zeros_like(self.kp)
        self.dv = torch.zeros_like(self.vp)

    def _keys(self, ks, vs, R):
        if ks is None:
            return self.kp, self.vp, torch.ones((R, self.kp.shape[0]), dtype=torch.bool)
        K = torch.cat([self.kp, ks[:, 0]])
        V = torch.cat([self.vp, vs[:, 0]])
        n = self.kp.shape[0]
        causal = torch.arange(R)[None, :] <= torch.arange(R)[:, None]
        mask = torch.cat([torch.ones((R, n), dtype=torch.bool), causal], dim=1)
        return K, V, mask

    def _fwd(self, q, ks, vs):
        K, V, mask = self._keys(ks, vs, q.shape[0])
        S = (self.s * q[:, 0] @ K.T).masked_fill(~mask, float("-inf"))
        m = S.amax(dim=1, keepdim=True)
        E = torch.exp(S - m)
        lse = m[:, 0] + torch.log(E.sum(dim=1))
        return (E @ V / E.sum(dim=1, keepdim=True))[:, None, :], lse[:, None]

    def _bwd(self, q, ks, vs, o, lse, do):
        K, V, mask = self._keys(ks, vs, q.shape[0])
        P = torch.exp(self.s * q[:, 0] @ K.T - lse) * mask
        dS = P * (do[:, 0] @ V.T - (do[:, 0] * o[:, 0]).sum(dim=1, keepdim=True))
        dk = self.s * dS.T @ q[:, 0]
        dv = P.T @ do[:, 0]
        n = self.kp.shape[0]
        self.dk += dk[:n]
        self.dv += dv[:n]
        return (self.s * dS @ K)[:, None, :], dk[n:, None, :], dv[n:, None, :]

    def fwd(self, q, ks, vs):
        self.calls.append("fwd")
        return self._fwd(q, ks, vs)

    def fwd_prompt_only(self, q):
        self.calls.append("fwd_prompt_only")
        return self._fwd(q, None, None)

    def bwd(self, q, ks, vs, o, lse, do):
        self.calls.append("bwd")
        return self._bwd(q, ks, vs, o, lse, do)

    def bwd_prompt_only(self, q, o, lse, do):
        self.calls.append("bwd_prompt_only")
        return self._bwd(q, None, None, o, lse, do)[0]


def _cp_replay_worker(rank, world, port, out):
    import torch.distributed as dist
    from long_context_grpo_gb300 import cp
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    kp, vp, q, ks, vs, do = _cp_inputs()
    b = cp.shard_bounds(kp.shape[0], world)
    pre = _ShardStandIn(kp[b[rank]:b[rank + 1]], vp[b[rank]:b[rank + 1]])
    o, lse, dq, dks, dvs = cp.replay_response(pre, rank, world, q, ks, vs, do, ops=_HostOps)
    out[rank] = dict(o=o.numpy(), lse=lse.numpy(), dq=dq.numpy(), calls=pre.calls,
                     dks=None if dks is None else dks.numpy(),
                     dvs=None if dvs is None else dvs.numpy(),
                     dk=pre.dk.numpy(), dv=pre.dv.numpy(), rows=(b[rank], b[rank + 1]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_context_parallel_replay_response_on_gloo_ranks(world):
    """cp.replay_response on gloo ranks (stand-ins for the shard kernels and the merge):
    only the last rank takes the suffix-owner path, the partials are merged in rank order,
    every rank ends with the same o, lse and dq, equal to the whole-prompt oracle replay,
    and each rank's prompt-key gradients are the oracle's rows of its own shard."""
    import numpy as np
    import oracle
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_cp_replay_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    kp, vp, q, ks, vs, do = _cp_inputs()
    ref = oracle.replay_response(kp, vp, q, ks, vs, do)
    for rank in range(world):
        r = res[rank]
        owner = rank == world - 1
        assert r["calls"] == (["fwd", "bwd"] if owner else ["fwd_prompt_only", "bwd_prompt_only"])
        np.testing.assert_allclose(r["o"], ref["o"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["lse"], ref["lse"], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["dq"], ref["dq"], rtol=0, atol=1e-12)
        a, b = r["rows"]
        np.testing.assert_allclose(r["dk"], ref["dk_prefix"][a:b, 0], rtol=0, atol=1e-12)
        np.testing.assert_allclose(r["dv"], ref["dv_prefix"][a:b, 0], rtol=0, atol=1e-12)
        if owner:
            np.testing.assert_allclose(r["dks"], ref["dk_suffix"], rtol=0, atol=1e-12)
            np.testing.assert_allclose(r["dvs"], ref["dv_suffix"], rtol=0, atol=1e-12)
        else:
            assert r["dks"] is None and r["dvs"] is None

"""The measurement code on the CPU: the algorithmic work formula, the traffic record's
source gating, and the reference arm's JSON line (every key the benchmark contract asks
for)."""
import json
import os

import pytest

import bench


def test_pairs_counts_visible_query_key_pairs():
    # brute force: suffix row t sees every prompt key and suffix keys 0..t
    for P in (0, 1, 5, 17):
        for R in (1, 2, 9):
            n = sum(1 for t in range(R) for j in range(P + R) if j < P or j - P <= t)
            assert bench.pairs(P, R) == n


def test_traffic_is_scaled_by_work_units_and_gated_by_the_source_hash(tmp_path, monkeypatch):
    """The dK/dV traffic record scales by 128-key work units, and only while the recorded
    hash equals the kernel source's (a stale record gives no number)."""
    import hashlib
    from long_context_grpo_gb300 import workloads as wl
    w = wl.WORKLOADS["p2m"]
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")))["bwd_dkdv"]
    src_bytes = open(os.path.join(bench.ROOT, rec["kernel_source"]), "rb").read()
    src = tmp_path / rec["kernel_source"]
    os.makedirs(src.parent, exist_ok=True)
    src.write_bytes(src_bytes)
    os.makedirs(tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    units = [w.Hkv * (w.P // 128 + 1), w.Hkv * (w.P // 128 + 2)]
    fresh = dict(rec, dram_bytes_per_unit=300000,
                 kernel_source_sha256_16=hashlib.sha256(src_bytes).hexdigest()[:16])
    json.dump({"bwd_dkdv": fresh}, open(tmp_path / "profiles" / "ncu_traffic.json", "w"))
    assert bench.load_traffic(w, [128, 256]) == pytest.approx(300000 * sum(units) / 2)
    stale = dict(fresh, kernel_source_sha256_16="0" * 16)
    json.dump({"bwd_dkdv": stale}, open(tmp_path / "profiles" / "ncu_traffic.json", "w"))
    assert bench.load_traffic(w, [128]) is None


def test_reference_arm_prints_one_complete_json_line(monkeypatch, capsys):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--workload", "tiny",
                                     "--steps", "1", "--warmup", "3", "--cpu-rows", "2"])
    bench.main()
    out = capsys.readouterr().out.strip().splitlines()
    assert len(out) == 1
    d = json.loads(out[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "tiny"


def test_warmup_below_three_is_refused(monkeypatch):
    monkeypatch.setattr("sys.argv", ["bench.py", "--warmup", "2"])
    with pytest.raises(SystemExit):
        bench.main()


def test_slow_staging_groups_are_replaced_at_most_twice():
    """The end-to-end harness replaces a pinned staging group that copies below half the best
    group's rate (kept aside, not freed) and gives up after two tries."""
    import bench
    groups = ["g0", "g1", "g2", "g3"]
    rates = [20.0, 211.0, 210.0, 30.0]
    # group 0 is fast once reallocated; group 3 stays slow
    next_rate = {0: [211.0], 3: [40.0, 35.0]}
    made = []

    def alloc(k):
        made.append(k)
        return "g%d'%d" % (k, len([m for m in made if m == k]))

    def rate(k):
        return next_rate[k].pop(0)

    aside, n = bench.replace_slow_groups(groups, rates, alloc, rate)
    assert n == 3 and made == [0, 3, 3]
    assert aside == ["g0", "g3", "g3'1"]
    assert groups == ["g0'1", "g1", "g2", "g3'2"]
    assert rates == [211.0, 211.0, 210.0, 35.0]

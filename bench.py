"""Benchmark of the branch-replay hot path on GB300.

One step = one GRPO group through the whole per-GPU hot path: prompt prepare (accumulator
zeroing), then for each of the G responses serially the forward replay, the fused GRPO
loss and the backward replay (prompt dK/dV accumulated in fp32), then the one prompt
gradient finalization.  Inputs are synthetic and seeded, with the shapes and distributions
of the workload table in long_context_grpo_gb300/workloads.py, resident in HBM before the
timed region (they are far larger than L2, so no flush is needed between steps).

Prints one JSON line.  `--impl reference` times the float64 CPU oracle instead, on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "branch-replay fwd+bwd TFLOP/s & response tok/s at P=2M; % of roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def pairs(P, R):
    """Visible (query, key) pairs of one response per query head."""
    return R * P + R * (R + 1) // 2


KERNELS_PER_BRACKET = {"zero": 2, "grpo_loss": 2, "finalize": 2}   # kernels one timed call launches


def load_traffic(w, R_list):
    """Per-launch DRAM traffic of the dK/dV kernel from the committed ncu capture, scaled by
    work units (128-key tiles); None once the profiled kernel source has changed."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            t = json.load(f)["bwd_dkdv"]
        src = os.path.join(ROOT, t["kernel_source"])
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if sha != t["kernel_source_sha256_16"]:
            return None
        units = [w.Hkv * ((w.P + 127) // 128 + (R + 127) // 128) for R in R_list]
        return t["dram_bytes_per_unit"] * sum(units) / len(units)
    except Exception:
        return None


def rank_max(x, dist=None, device="cpu"):
    """Max of a per-rank scalar over all ranks (the job's time is its slowest rank's)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_sum(x, dist=None, device="cpu"):
    """Sum of a per-rank scalar over all ranks (whole-job work)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t)
    return float(t.item())


def load_peaks():
    """The measured peaks (copy bandwidth, cuBLAS bf16 burst and sustained) and the
    median SM clock under load while they were measured (None if not recorded)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        peaks = {k: float(d[k]) for k in FALLBACK_PEAKS}
        peaks["sm_mhz"] = (d.get("clocks_under_load") or {}).get("sm_mhz_median")
        return peaks, "measured"
    except Exception:
        out = dict(FALLBACK_PEAKS)
        out["sm_mhz"] = None
        return out, "fallback"


# Dense bf16 tensor figures of the GPU, for context beside the measured peaks: NVIDIA's
# nominal dense bf16 rate, and the tensor pipe's issue rate (8192 bf16 FLOP per clock per SM
# for the 128 x N x 16 instruction shapes used here) at the clock a run actually held.
NOMINAL_DENSE_BF16_TFLOPS = 2250.0
TENSOR_FLOP_PER_CLK_PER_SM = 8192


def tensor_context(achieved, peaks, run_mhz, n_sms):
    """Fractions of a contraction's achieved TFLOP/s against other denominators than the
    contract's sustained cuBLAS figure: the cuBLAS burst figure, the nominal dense rate, the
    tensor pipe at the run's median clock, and the sustained figure rescaled to the run's
    clock (the peak was measured under the power cap at a lower clock)."""
    out = {"frac_of_burst": achieved / peaks["bf16_tflops"],
           "frac_of_nominal_dense": achieved / NOMINAL_DENSE_BF16_TFLOPS,
           "run_sm_mhz": run_mhz, "peak_sm_mhz": peaks.get("sm_mhz")}
    if run_mhz:
        pipe = TENSOR_FLOP_PER_CLK_PER_SM * n_sms * run_mhz * 1e6 / 1e12
        out["tensor_pipe_tflops_at_run_clock"] = pipe
        out["frac_of_tensor_pipe_at_run_clock"] = achieved / pipe
        if peaks.get("sm_mhz"):
            out["frac_of_sustained_per_clock"] = (achieved / run_mhz) / (
                peaks["bf16_tflops_sustained"] / peaks["sm_mhz"])
    return out


# ------------------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.proc = None
        self.sel = None
        try:
            import torch
            props = torch.cuda.get_device_properties(device_index)
            uuid = getattr(props, "uuid", None)
            if uuid is not None:
                self.sel = "GPU-%s" % uuid
        except Exception:
            self.sel = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.sel:
            cmd += ["-i", self.sel]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------------------ CPU side
def cpu_sample_inputs(w, seed, rows):
    """Inputs of the bounded CPU sample: the full prompt of one kv head and the first `rows`
    query rows of response 0 for one query head (same distributions as the workload)."""
    from long_context_grpo_gb300 import workloads as wl
    import dataclasses
    w1 = dataclasses.replace(w, Hq=1, Hkv=1)
    kp, vp = wl.prefix_kv(w1, seed, "cpu")
    q, ks, vs, do = wl.response_attention(w1, 0, rows, seed, "cpu")
    logits, ids, noise = wl.response_loss_inputs(w, 0, rows, seed, "cpu")
    return kp, vp, q, ks, vs, do, logits, ids, noise


def oracle_sample_step(w, inp, G):
    """One bounded oracle step: fwd + bwd of `rows` query rows x 1 head against the full
    prompt, plus the GRPO loss of those rows.  Returns algorithmic FLOPs of the sample."""
    import oracle
    kp, vp, q, ks, vs, do, logits, ids, noise = inp
    rows = q.shape[0]
    oracle.replay_response(kp, vp, q, ks, vs, do)
    logp = oracle.token_logp(logits, ids)
    oracle.grpo_loss(logits, ids, logp + noise.double().numpy(), 1.0, w.eps, G)
    return 14 * w.D * pairs(w.P, rows)


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def run_reference(args, w):
    """The float64 oracle, as it stands, on the host cores: W warm-up + K timed steps of a
    bounded sample of the workload."""
    rows = args.cpu_rows
    inp = cpu_sample_inputs(w, args.seed, rows)
    for _ in range(args.warmup):
        oracle_sample_step(w, inp, w.G)
    t0 = time.perf_counter()
    flops = 0
    for _ in range(args.steps):
        flops += oracle_sample_step(w, inp, w.G)
    dt = time.perf_counter() - t0
    tflops = flops / dt / 1e12
    tok_s = args.steps * rows / w.Hq / dt
    sample = ("float64 oracle: %d query rows x 1 of %d query heads of response 0 against the "
              "full %d-token prompt (fwd + bwd), plus their GRPO loss over V=%d; "
              "tok/s = rows / Hq per second" % (rows, w.Hq, w.P, w.V))
    line = {"metric": METRIC, "value": tflops, "unit": "TFLOP/s", "impl": "reference",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "P": w.P, "G": w.G, "Hq": w.Hq, "Hkv": w.Hkv,
                       "D": w.D, "V": w.V, "sample_rows": rows},
            "response_tok_s": tok_s,
            "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------------------ GPU side
class Group:
    """Device-resident inputs and reusable output buffers of one group."""

    def __init__(self, w, seed, device):
        import torch
        import long_context_grpo_gb300 as ls
        from long_context_grpo_gb300 import workloads as wl
        self.w = w
        self.R = wl.response_lengths(w, seed)
        self.A = wl.group_advantages(wl.rewards(w, seed))
        if all(a == 0.0 for a in self.A):      # degenerate draw: keep the loss path non-trivial
            self.A = wl.group_advantages([float(i % 2) for i in range(w.G)])
        self.kp, self.vp = wl.prefix_kv(w, seed, device)
        self.resp = []
        for i, Ri in enumerate(self.R):
            q, ks, vs, do = wl.response_attention(w, i, Ri, seed, device)
            logits, ids, noise = wl.response_loss_inputs(w, i, Ri, seed, device)
            self.resp.append({"q": q, "ks": ks, "vs": vs, "do": do, "logits": logits,
                              "ids": ids, "noise": noise, "old": None})
        Rm = max(self.R)
        f32, bf16 = torch.float32, torch.bfloat16
        self.dk_acc = torch.empty(self.kp.shape, dtype=f32, device=device)
        self.dv_acc = torch.empty(self.kp.shape, dtype=f32, device=device)
        self.dk_out = torch.empty(self.kp.shape, dtype=bf16, device=device)
        self.dv_out = torch.empty(self.kp.shape, dtype=bf16, device=device)
        self.o = torch.empty((Rm, w.Hq, w.D), dtype=bf16, device=device)
        self.lse = torch.empty((Rm, w.Hq), dtype=f32, device=device)
        self.dq = torch.empty((Rm, w.Hq, w.D), dtype=bf16, device=device)
        self.dks = torch.empty((Rm, w.Hkv, w.D), dtype=bf16, device=device)
        self.dvs = torch.empty((Rm, w.Hkv, w.D), dtype=bf16, device=device)
        self.dlog = torch.empty((Rm, w.V), dtype=bf16, device=device)
        self.mask = torch.empty((Rm,), dtype=torch.uint8, device=device)
        self.logp = torch.empty((Rm,), dtype=f32, device=device)
        self.lws = torch.empty(ls.grpo_loss_workspace_bytes(Rm), dtype=torch.uint8, device=device)
        pre = ls.Prefix(self.kp, self.vp, self.dk_acc, self.dv_acc, Hq=w.Hq)
        self.bws = torch.empty(max(pre.bwd_workspace_bytes(Rm), 16), dtype=torch.uint8,
                               device=device)
        # old-policy log-probs: the current policy's token log-prob plus the drawn noise
        scratch = torch.zeros(1, dtype=torch.float64, device=device)
        for r, Ri in zip(self.resp, self.R):
            zero_old = torch.zeros((Ri,), dtype=f32, device=device)
            ls.grpo_loss(r["logits"], r["ids"], zero_old, 0.0, w.eps, w.G, scratch,
                         dlogits=self.dlog[:Ri], clip_mask=self.mask[:Ri],
                         logp_out=self.logp[:Ri], workspace=self.lws)
            r["old"] = self.logp[:Ri] + r["noise"]
        pre.close()
        torch.cuda.synchronize()

    def input_groups(self):
        """Device inputs of one step in the order a step consumes them: the prompt K/V, then
        each response's tensors."""
        out = [[self.kp, self.vp]]
        for r in self.resp:
            out.append([r["q"], r["ks"], r["vs"], r["do"], r["logits"], r["ids"], r["old"]])
        return out

    def step(self, loss_slot, ev_in=None, ev_used=None, out=None):
        """One group step.  With events (end-to-end runs): input group k is waited for
        (ev_in[k]) before its first use and ev_used[k] is recorded after its last use, so
        the copies of later responses overlap the replay of earlier ones.  With `out` (a
        HostResults), each response's results and the finalized prompt gradient are copied
        back to the host as soon as they are written, overlapping the rest of the step."""
        import torch
        import long_context_grpo_gb300 as ls
        w = self.w
        cur = torch.cuda.current_stream()
        if ev_in is not None:
            cur.wait_event(ev_in[0])
        pre = ls.Prefix(self.kp, self.vp, self.dk_acc, self.dv_acc, Hq=w.Hq)
        for i, (r, Ri) in enumerate(zip(self.resp, self.R)):
            if ev_in is not None:
                cur.wait_event(ev_in[1 + i])
            o, lse = pre.fwd(r["q"], r["ks"], r["vs"], o=self.o[:Ri], lse=self.lse[:Ri])
            if out is not None:
                out.before_response(cur)
            ls.grpo_loss(r["logits"], r["ids"], r["old"], self.A[i], w.eps, w.G, loss_slot,
                         dlogits=self.dlog[:Ri], clip_mask=self.mask[:Ri],
                         logp_out=self.logp[:Ri], workspace=self.lws)
            pre.bwd(r["q"], r["ks"], r["vs"], o, lse, r["do"], dq=self.dq[:Ri],
                    dk_suffix=self.dks[:Ri], dv_suffix=self.dvs[:Ri], workspace=self.bws)
            if ev_used is not None:
                ev_used[1 + i].record(cur)
            if out is not None:
                out.response_done(i, cur)
        if ev_used is not None:
            ev_used[0].record(cur)
        if out is not None:
            out.before_finalize(cur)
        pre.finalize(1.0, self.dk_out, self.dv_out)
        if out is not None:
            out.finalize_done(cur)
        pre.close()

    def score(self):
        """Old/reference-policy scoring of the group: forward replay + token log-probs."""
        import long_context_grpo_gb300 as ls
        pre = ls.Prefix(self.kp, self.vp, self.dk_acc, self.dv_acc, Hq=self.w.Hq)
        for r, Ri in zip(self.resp, self.R):
            pre.fwd(r["q"], r["ks"], r["vs"], o=self.o[:Ri], lse=self.lse[:Ri])
            ls.token_logp(r["logits"], r["ids"], logp_out=self.logp[:Ri])
        pre.close()

    def block_replay(self, block, stream):
        """Blockwise suffix replay of the group's longest response (fwd of every block, then
        bwd of every block in reverse) against the whole-response replay of the same rows;
        both timed with CUDA events on `stream`, after one untimed run each."""
        import torch
        import long_context_grpo_gb300 as ls
        w = self.w
        i = max(range(len(self.R)), key=lambda k: self.R[k])
        R, r = self.R[i], self.resp[i]
        P0, dev = w.P, self.kp.device
        kbuf = torch.empty((P0 + R, w.Hkv, w.D), dtype=torch.bfloat16, device=dev)
        vbuf = torch.empty_like(kbuf)
        kbuf[:P0] = self.kp
        kbuf[P0:] = r["ks"]
        vbuf[:P0] = self.vp
        vbuf[P0:] = r["vs"]
        dk = torch.empty(kbuf.shape, dtype=torch.float32, device=dev)
        dv = torch.empty_like(dk)
        spans = [(t0, min(R, t0 + block)) for t0 in range(0, R, block)]
        q, do = r["q"], r["do"]
        o, lse, dq = self.o[:R], self.lse[:R], self.dq[:R]

        def blocks(pre):
            for t0, t1 in spans:
                pre.block_fwd(P0 + t0, q[t0:t1], o[t0:t1], lse[t0:t1])
            for t0, t1 in reversed(spans):
                pre.block_bwd(P0 + t0, q[t0:t1], o[t0:t1], lse[t0:t1], do[t0:t1], dq[t0:t1],
                              workspace=self.bws)

        def whole(pre):
            pre.fwd(q, r["ks"], r["vs"], o=o, lse=lse)
            pre.bwd(q, r["ks"], r["vs"], o, lse, do, dq=dq, dk_suffix=self.dks[:R],
                    dv_suffix=self.dvs[:R], workspace=self.bws)

        def timed(fn, pre):
            fn(pre)
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(pre)
            e1.record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)

        pb = ls.Prefix(kbuf, vbuf, dk, dv, Hq=w.Hq)
        ms_b = timed(blocks, pb)
        pb.close()
        pw = ls.Prefix(self.kp, self.vp, self.dk_acc, self.dv_acc, Hq=w.Hq)
        ms_w = timed(whole, pw)
        pw.close()
        del kbuf, vbuf, dk, dv
        fl = 14 * w.D * w.Hq * pairs(P0, R)
        act = lambda n: n * w.Hq * (4 * w.D * 2 + 4)   # q, o, dO, dq (bf16) and lse per row
        return {"response_tokens": R, "block": block, "blocks": len(spans),
                "ms": ms_b, "tflops": fl / (ms_b / 1e3) / 1e12,
                "whole_response_ms": ms_w, "whole_response_tflops": fl / (ms_w / 1e3) / 1e12,
                "attention_activation_bytes_per_block": act(min(block, R)),
                "attention_activation_bytes_whole": act(R)}

    def packed_replay(self, stream, loss_slot):
        """The group as one packed (tree) replay: one forward launch for all responses, the
        G loss calls, one backward launch, one finalize; timed like the serial step after one
        untimed run.  Returns its time and the extra activation memory it holds."""
        import torch
        import long_context_grpo_gb300 as ls
        w = self.w
        cu = [0]
        for Ri in self.R:
            cu.append(cu[-1] + Ri)
        q, ks, vs, do = (torch.cat([r[k] for r in self.resp]) for k in ("q", "ks", "vs", "do"))
        T = cu[-1]
        o = torch.empty_like(q)
        lse = torch.empty((T, w.Hq), dtype=torch.float32, device=q.device)
        dq = torch.empty_like(q)
        dks = torch.empty_like(ks)
        dvs = torch.empty_like(vs)

        def step():
            pre = ls.Prefix(self.kp, self.vp, self.dk_acc, self.dv_acc, Hq=w.Hq)
            pre.fwd_packed(cu, q, ks, vs, o=o, lse=lse)
            for i, (r, Ri) in enumerate(zip(self.resp, self.R)):
                ls.grpo_loss(r["logits"], r["ids"], r["old"], self.A[i], w.eps, w.G, loss_slot,
                             dlogits=self.dlog[:Ri], clip_mask=self.mask[:Ri],
                             logp_out=self.logp[:Ri], workspace=self.lws)
            pre.bwd_packed(cu, q, ks, vs, o, lse, do, dq=dq, dk_suffix=dks, dv_suffix=dvs)
            pre.finalize(1.0, self.dk_out, self.dv_out)
            pre.close()

        step()
        torch.cuda.synchronize()
        ls.timing_read()
        ls.timing_enable(True)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        ls.timing_enable(False)
        kt = ls.timing_read()
        ms = e0.elapsed_time(e1)
        extra = sum(t.numel() * t.element_size() for t in (q, ks, vs, do, o, lse, dq, dks, dvs))
        del q, ks, vs, do, o, lse, dq, dks, dvs
        return {"ms": ms, "tflops": self.flops() / (ms / 1e3) / 1e12,
                "response_tok_s": sum(self.R) / (ms / 1e3), "launches_attention": 2 + 3,
                "kernel_ms": {k: round(v[0], 3) for k, v in kt.items() if v[1] > 0},
                "activation_bytes_held": extra}

    def cp_replay(self, shards, stream):
        """Context-parallel replay of the longest response with the prompt split into
        `shards` contiguous shards (one handle each; the last also owns the causal suffix):
        partial forwards, merge, shard backwards with the merged O/LSE, dQ part sum.  The
        ranks are emulated on this GPU; timed after one untimed run."""
        import torch
        import long_context_grpo_gb300 as ls
        w = self.w
        i = max(range(len(self.R)), key=lambda k: self.R[k])
        R, r = self.R[i], self.resp[i]
        q, ks, vs, do = r["q"], r["ks"], r["vs"], r["do"]
        bounds = [round(k * w.P / shards) for k in range(shards + 1)]
        hs = [ls.Prefix(self.kp[a:b], self.vp[a:b], self.dk_acc[a:b], self.dv_acc[a:b], Hq=w.Hq)
              for a, b in zip(bounds[:-1], bounds[1:])]
        o_parts = [torch.empty_like(q) for _ in hs]
        lse_parts = [torch.empty((R, w.Hq), dtype=torch.float32, device=q.device) for _ in hs]
        dq_parts = [torch.empty_like(q) for _ in hs]
        o, lse, dq = self.o[:R], self.lse[:R], self.dq[:R]

        def run():
            for h, op, lp in zip(hs[:-1], o_parts, lse_parts):
                h.fwd_prompt_only(q, op, lp)
            hs[-1].fwd(q, ks, vs, o=o_parts[-1], lse=lse_parts[-1])
            ls.attn_merge(o_parts, lse_parts, o=o, lse=lse)
            for h, dp in zip(hs[:-1], dq_parts):
                h.bwd_prompt_only(q, o, lse, do, dq=dp, workspace=self.bws)
            hs[-1].bwd(q, ks, vs, o, lse, do, dq=dq_parts[-1], dk_suffix=self.dks[:R],
                       dv_suffix=self.dvs[:R], workspace=self.bws)
            ls.sum_bf16(dq_parts, out=dq)

        run()
        torch.cuda.synchronize()
        ls.timing_read()
        ls.timing_enable(True)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run()
        e1.record(stream)
        torch.cuda.synchronize()
        ls.timing_enable(False)
        kt = ls.timing_read()
        for h in hs:
            h.close()
        ms = e0.elapsed_time(e1)
        fl = 14 * w.D * w.Hq * pairs(w.P, R)
        row = R * w.Hq
        merge_bytes = shards * row * (2 * w.D + 4) + row * (2 * w.D + 4)
        sum_bytes = (shards + 1) * row * 2 * w.D
        mm, sm = kt["merge"][0], kt["sum"][0]
        return {"shards": shards, "response_tokens": R, "ms": ms,
                "tflops": fl / (ms / 1e3) / 1e12,
                "merge_ms": mm, "merge_gbs": merge_bytes / (mm / 1e3) / 1e9 if mm > 0 else None,
                "sum_ms": sm, "sum_gbs": sum_bytes / (sm / 1e3) / 1e9 if sm > 0 else None,
                "note": "shards emulated as separate handles on one GPU; the collectives "
                        "(all-gather of partials, reduce of dQ) are not run"}

    def flops(self):
        w = self.w
        return sum(14 * w.D * w.Hq * pairs(w.P, Ri) for Ri in self.R)

    def kernel_work(self):
        """Algorithmic work per kernel id for one step: (amount, unit)."""
        w = self.w
        pr = sum(pairs(w.P, Ri) for Ri in self.R)
        n = w.P * w.Hkv * w.D
        return {
            "replay_fwd": (4 * w.D * w.Hq * pr, "flop"),
            "bwd_dkdv": (8 * w.D * w.Hq * pr, "flop"),
            "bwd_dq": (2 * w.D * w.Hq * pr, "flop"),
            "grpo_loss": (sum(Ri * (4 * w.V + 12) for Ri in self.R), "byte"),
            "bwd_prep": (sum(Ri * w.Hq * (4 * w.D + 4) for Ri in self.R), "byte"),
            "finalize": (2 * n * 6, "byte"),
            "zero": (2 * n * 4, "byte"),
        }


def replace_slow_groups(groups, rates, alloc, rate, tries=2, frac=0.5):
    """Reallocate each staging group whose copy rate is below `frac` of the best group's,
    at most `tries` times per group.  groups / rates are updated in place; alloc(k) returns a
    new group k, rate(k) measures group k as it now stands.  The replaced groups are returned
    (the caller keeps them alive, so that the allocator does not hand the same block back)
    with the number of reallocations."""
    set_aside, realloc = [], 0
    for k in range(len(groups)):
        for _ in range(tries):
            if rates[k] >= frac * max(rates):
                break
            set_aside.append(groups[k])
            groups[k] = alloc(k)
            rates[k] = rate(k)
            realloc += 1
    return set_aside, realloc


class HostResults:
    """Pinned host copies of one step's results, filled on a copy stream while the step
    runs: per response dQ, suffix dK/dV, clip mask and token log-prob (as soon as that
    response's backward has written them), and the finalized prompt dK/dV at the end.  The
    compute stream reuses the device buffers only after the previous copy out of them has
    completed.  dlogits stay on the device (they feed the LM-head backward there)."""

    def __init__(self, grp, copy_stream):
        import torch
        self.grp, self.cs = grp, copy_stream
        w = grp.w

        def pin(shape, dtype):
            return torch.empty(shape, dtype=dtype, pin_memory=True)

        self.resp = [{"dq": pin((Ri, w.Hq, w.D), torch.bfloat16),
                      "dks": pin((Ri, w.Hkv, w.D), torch.bfloat16),
                      "dvs": pin((Ri, w.Hkv, w.D), torch.bfloat16),
                      "mask": pin((Ri,), torch.uint8), "logp": pin((Ri,), torch.float32)}
                     for Ri in grp.R]
        self.dk = pin(tuple(grp.dk_out.shape), torch.bfloat16)
        self.dv = pin(tuple(grp.dv_out.shape), torch.bfloat16)
        self.bytes = sum(t.numel() * t.element_size() for d in self.resp for t in d.values())
        self.bytes += 2 * self.dk.numel() * self.dk.element_size()
        self.resp_copied = None     # copy of the last response's outputs finished
        self.fin_copied = None      # copy of the finalized prompt gradient finished

    def before_response(self, cur):
        if self.resp_copied is not None:
            cur.wait_event(self.resp_copied)

    def response_done(self, i, cur):
        import torch
        g, Ri = self.grp, self.grp.R[i]
        ready = torch.cuda.Event()
        ready.record(cur)
        self.cs.wait_event(ready)
        h = self.resp[i]
        with torch.cuda.stream(self.cs):
            h["dq"].copy_(g.dq[:Ri], non_blocking=True)
            h["dks"].copy_(g.dks[:Ri], non_blocking=True)
            h["dvs"].copy_(g.dvs[:Ri], non_blocking=True)
            h["mask"].copy_(g.mask[:Ri], non_blocking=True)
            h["logp"].copy_(g.logp[:Ri], non_blocking=True)
        self.resp_copied = torch.cuda.Event()
        self.resp_copied.record(self.cs)

    def before_finalize(self, cur):
        if self.fin_copied is not None:
            cur.wait_event(self.fin_copied)

    def finalize_done(self, cur):
        import torch
        ready = torch.cuda.Event()
        ready.record(cur)
        self.cs.wait_event(ready)
        with torch.cuda.stream(self.cs):
            self.dk.copy_(self.grp.dk_out, non_blocking=True)
            self.dv.copy_(self.grp.dv_out, non_blocking=True)
        self.fin_copied = torch.cuda.Event()
        self.fin_copied.record(self.cs)


def time_group(grp, steps, warmup, stream, peaks, n_sms, losses):
    """Warm-up and timed steps of one group on this GPU (CUDA events on `stream`, every
    library launch timed on its own stream): (ms per step, per-kernel table)."""
    import torch
    import long_context_grpo_gb300 as ls
    for k in range(warmup):
        grp.step(losses[k % losses.numel():k % losses.numel() + 1])
    torch.cuda.synchronize()
    ls.timing_read()
    ls.timing_enable(True)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        grp.step(losses[k % losses.numel():k % losses.numel() + 1])
    e1.record(stream)
    torch.cuda.synchronize()
    ls.timing_enable(False)
    kt = ls.timing_read()
    ms = e0.elapsed_time(e1)
    return ms / steps, kernel_table(kt, grp.kernel_work(), steps, ms, peaks)


def kernel_table(kt, work, steps, total_ms, peaks):
    """Per kernel: launches, average ms, share of the timed region, achieved rate against
    the measured peak of its bound (sustained bf16 for contractions, HBM copy otherwise)."""
    kernels = {}
    for name, (tot_ms, n) in kt.items():
        if n == 0 or tot_ms <= 0 or name not in work:
            continue
        amount, unit = work[name]
        per_launch_amount = amount * steps / n
        avg_ms = tot_ms / n
        if unit == "flop":
            ach = per_launch_amount / (avg_ms / 1e3) / 1e12
            pk, pu, bound = peaks["bf16_tflops_sustained"], "TFLOP/s", "tensor"
        else:
            ach = per_launch_amount / (avg_ms / 1e3) / 1e9
            pk, pu, bound = peaks["hbm_gbs"], "GB/s", "hbm"
        kernels[name] = {"launches": n, "avg_ms": avg_ms, "share": tot_ms / total_ms,
                         "bound": bound, "achieved": ach, "peak": pk, "unit": pu,
                         "frac": ach / pk}
    return kernels


def measure_configs(names, args, dev, stream, peaks, n_sms):
    """Throughput of the whole group step on the other workload configurations (the same
    step, launch configuration and timing as the headline measurement), one at a time."""
    import torch
    from long_context_grpo_gb300 import workloads as wl
    out = {}
    losses = torch.zeros(4, dtype=torch.float64, device=dev)
    for name in names:
        w = wl.WORKLOADS[name]
        grp = Group(w, args.seed, dev)
        ms, kernels = time_group(grp, args.config_steps, args.warmup, stream, peaks, n_sms,
                                 losses)
        out[name] = {"value": grp.flops() / (ms / 1e3) / 1e12, "unit": "TFLOP/s",
                     "response_tok_s": sum(grp.R) / (ms / 1e3), "ms_per_step": ms,
                     "steps": args.config_steps, "P": w.P, "G": w.G, "R": grp.R,
                     "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "V": w.V,
                     "kernels": {k: {"frac": round(v["frac"], 4), "achieved": round(v["achieved"], 1),
                                     "unit": v["unit"], "share": round(v["share"], 4)}
                                 for k, v in kernels.items()}}
        del grp
        torch.cuda.empty_cache()
    return out


def run_ours(args, w):
    import torch
    import long_context_grpo_gb300 as ls

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    def barrier():
        if dist is not None:
            dist.barrier()

    def max_over_ranks(x):
        return rank_max(x, dist, dev)

    def sum_over_ranks(x):
        return rank_sum(x, dist, dev)

    grp = Group(w, args.seed + rank, dev)
    losses = torch.zeros(args.warmup + 2 * args.steps + 2, dtype=torch.float64, device=dev)
    slot = 0
    for _ in range(args.warmup):
        grp.step(losses[slot:slot + 1])
        slot += 1
    torch.cuda.synchronize()
    st = ls.device_status()
    if st != (0, 0):
        raise RuntimeError("device status after warm-up: %s" % (st,))

    # ---------------- device-resident timed region
    stream = torch.cuda.current_stream()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index)
    ls.timing_read()
    ls.timing_enable(True)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    ev0.record(stream)
    for _ in range(args.steps):
        grp.step(losses[slot:slot + 1])
        slot += 1
    ev1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ls.timing_enable(False)
    kt = ls.timing_read()
    barrier()
    ms = ev0.elapsed_time(ev1)
    ms_max = max_over_ranks(ms)
    flops_all = sum_over_ranks(grp.flops() * args.steps)
    toks_all = sum_over_ranks(sum(grp.R) * args.steps)
    value = flops_all / (ms_max / 1e3) / 1e12
    tok_s = toks_all / (ms_max / 1e3)
    st = ls.device_status()
    if st != (0, 0):
        raise RuntimeError("device status after timed steps: %s" % (st,))

    # ---------------- per-kernel roofline
    peaks, peak_src = load_peaks()
    n_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    kernels = kernel_table(kt, grp.kernel_work(), args.steps, ms, peaks)
    for name, kd in kernels.items():
        if kd["bound"] == "tensor":
            kd.update(tensor_context(kd["achieved"], peaks, clk.get("sm_mhz"), n_sms))
    dom = max(kernels, key=lambda k: kernels[k]["share"])
    d = kernels[dom]
    traffic = load_traffic(w, grp.R) if dom == "bwd_dkdv" else None
    roofline = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"],
                "unit": d["unit"], "frac": d["frac"], "traffic": traffic,
                "peak_source": peak_src + (" sustained bf16" if d["bound"] == "tensor" else " HBM copy")}
    if d["bound"] == "tensor":
        roofline.update({k: d[k] for k in d if k.startswith("frac_of") or k.endswith("mhz")
                         or k.startswith("tensor_pipe")})
    # the whole step (all kernels, algorithmic FLOPs) against the same denominators
    step_context = tensor_context(value, peaks, clk.get("sm_mhz"), n_sms)
    step_context["frac_of_sustained"] = value / peaks["bf16_tflops_sustained"]
    launches = sum(v["launches"] * KERNELS_PER_BRACKET.get(k, 1) for k, v in kernels.items())

    # ---------------- old/reference-policy scoring of the same group (no gradients)
    score = None
    if not args.no_score:
        grp.score()   # untimed
        torch.cuda.synchronize()
        ls.timing_read()
        ls.timing_enable(True)
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        grp.score()
        s1.record(stream)
        torch.cuda.synchronize()
        ls.timing_enable(False)
        st_k = ls.timing_read()
        sms = s0.elapsed_time(s1)
        fwd_flops = sum(4 * w.D * w.Hq * pairs(w.P, Ri) for Ri in grp.R)
        lp_ms, lp_n = st_k["token_logp"]
        lp_bytes = sum(Ri * (2 * w.V + 8) for Ri in grp.R)
        score = {"ms": sms, "fwd_tflops": fwd_flops / (sms / 1e3) / 1e12,
                 "response_tok_s": sum(grp.R) / (sms / 1e3),
                 "token_logp": {"launches": lp_n, "avg_ms": lp_ms / max(lp_n, 1),
                                "achieved_gbs": lp_bytes / (lp_ms / 1e3) / 1e9 if lp_ms > 0 else None,
                                "frac_hbm": (lp_bytes / (lp_ms / 1e3) / 1e9) / peaks["hbm_gbs"] if lp_ms > 0 else None}}

    # ---------------- blockwise suffix replay of the longest response
    blk = None
    if args.block > 0 and rank == 0:
        blk = grp.block_replay(args.block, stream)

    # ---------------- the group as one packed (tree) replay
    packed = None
    if not args.no_packed and rank == 0:
        packed = grp.packed_replay(stream, losses[0:1])
        packed["vs_serial_step"] = packed["ms"] and (ms / args.steps) / packed["ms"]

    # ---------------- context-parallel replay of the longest response (shards on this GPU)
    cp = None
    if args.cp_shards > 0 and rank == 0:
        cp = grp.cp_replay(args.cp_shards, stream)

    # ---------------- end to end through the C ABI with host buffers
    e2e = None
    if not args.no_e2e:
        # Each step copies every input from pinned host memory: the prompt K/V first, then
        # each response's tensors, on a copy stream, so that response i+1 is copied while
        # response i is replayed; a buffer is overwritten only after its last use.
        # The pinned staging buffers are allocated once.  On this machine the first large
        # pinned allocation of a process can come back at a tenth of the link's copy rate
        # (measured 20-37 GB/s against 211 GB/s for every later buffer, the same shape and
        # kind); a group copying below half the best group's rate is set aside (kept alive,
        # so that the allocator does not hand the same block back) and allocated again, at
        # most twice.  The per-group rates and the reallocations are in the e2e record.
        dev_groups = grp.input_groups()

        def alloc_group(g_):
            hg = []
            for t in g_:
                h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                h.copy_(t)
                hg.append(h)
            return hg

        def copy_gbs(hg, dg):
            torch.cuda.synchronize()
            c0 = torch.cuda.Event(enable_timing=True)
            c1 = torch.cuda.Event(enable_timing=True)
            c0.record()
            for h, d_ in zip(hg, dg):
                d_.copy_(h, non_blocking=True)
            c1.record()
            torch.cuda.synchronize()
            nb = sum(h.numel() * h.element_size() for h in hg)
            return nb / (c0.elapsed_time(c1) / 1e3) / 1e9

        host_groups = [alloc_group(g_) for g_ in dev_groups]
        rates = [copy_gbs(hg, dg) for hg, dg in zip(host_groups, dev_groups)]
        set_aside, realloc = replace_slow_groups(
            host_groups, rates, lambda k: alloc_group(dev_groups[k]),
            lambda k: copy_gbs(host_groups[k], dev_groups[k]))
        h2d = sum(t.numel() * t.element_size() for hg in host_groups for t in hg)
        host_loss = torch.empty(1, dtype=torch.float64).pin_memory()
        copy_stream = torch.cuda.Stream()      # host -> device, in consumption order
        back_stream = torch.cuda.Stream()      # device -> host, as results are written
        results = HostResults(grp, back_stream)
        ev_in = [torch.cuda.Event() for _ in dev_groups]
        ev_used = [torch.cuda.Event() for _ in dev_groups]
        steps_done = [0]

        def e2e_step():
            for k, (hg, dg) in enumerate(zip(host_groups, dev_groups)):
                if steps_done[0] > 0:
                    copy_stream.wait_event(ev_used[k])
                with torch.cuda.stream(copy_stream):
                    for h, d_ in zip(hg, dg):
                        d_.copy_(h, non_blocking=True)
                ev_in[k].record(copy_stream)
            grp.step(losses[slot:slot + 1], ev_in=ev_in, ev_used=ev_used, out=results)
            host_loss.copy_(losses[slot:slot + 1], non_blocking=True)
            steps_done[0] += 1

        e2e_step()   # untimed
        torch.cuda.synchronize()
        barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        ls.timing_read()
        ls.timing_enable(True)
        e0.record(stream)
        copy_stream.wait_event(e0)
        back_stream.wait_event(e0)
        for _ in range(args.steps):
            e2e_step()
        stream.wait_event(results.fin_copied)   # the last read-back is inside the timed region
        e1.record(stream)
        torch.cuda.synchronize()
        ls.timing_enable(False)
        e2e_k = ls.timing_read()
        ems = max_over_ranks(e0.elapsed_time(e1))
        e2e = {"value": flops_all / (ems / 1e3) / 1e12, "unit": "TFLOP/s",
               "response_tok_s": toks_all / (ems / 1e3), "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": results.bytes + 8,
               "d2h": "per response dQ, suffix dK/dV, clip mask and token log-prob, the "
                      "finalized bf16 prompt dK/dV and the fp64 loss; dlogits stay on the device",
               "kernel_ms_per_step": {k: round(v[0] / args.steps, 2) for k, v in e2e_k.items() if v[1] > 0},
               "h2d_gbs_per_group": [round(r, 1) for r in rates],
               "host_groups_reallocated": realloc}
        del host_groups, results, set_aside

    # ---------------- CPU baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # timed as the reference arm times it: warm-up samples, then several timed samples
        rows = args.cpu_rows
        inp = cpu_sample_inputs(w, args.seed, rows)
        for _ in range(args.cpu_warmup):
            oracle_sample_step(w, inp, w.G)
        t0 = time.perf_counter()
        fl = 0
        for _ in range(args.cpu_steps):
            fl += oracle_sample_step(w, inp, w.G)
        dt = time.perf_counter() - t0
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
               "sample": "float64 oracle, %d query rows x 1 of %d query heads of response 0 "
                         "against the full %d-token prompt (fwd + bwd) plus their GRPO loss; "
                         "%d warm-up + %d timed samples, %.1f s timed"
                         % (rows, w.Hq, w.P, args.cpu_warmup, args.cpu_steps, dt)}

    # ---------------- the other workload configurations (rank 0, whole group step each)
    configs = None
    names = [n for n in args.configs.split(",") if n and n != w.name]
    if names and rank == 0:
        configs = measure_configs(names, args, dev, stream, peaks, n_sms)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": w.name, "P": w.P, "G": w.G,
                           "R": grp.R if world == 1 else "per-rank draws",
                           "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D, "V": w.V,
                           "parallelism": "independent groups per GPU" if world > 1 else "1 GPU",
                           "l2": "inputs larger than L2 (no flush)"},
                "response_tok_s": tok_s,
                "roofline": roofline,
                "step_vs_peaks": step_context,
                "kernels": kernels,
                "gpu_launches": launches,
                "clocks": clk,
                "e2e": e2e,
                "cpu_baseline": cpu,
                "scoring": score,
                "block_replay": blk,
                "packed_replay": packed,
                "cp_replay": cp,
                "other_configs": configs,
                "receipt": {"gradient_semantics": "prompt dK/dV exposed (fp32, group-summed), "
                                                  "not propagated",
                            "residency": "prompt K/V resident in HBM for the group",
                            "topology": "%d GPU(s), no collective" % world,
                            "staleness": "none (prepared every step)"}}
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


def run_loss_only(args):
    """The GRPO loss and token log-prob kernels alone on one synthetic response of R rows of
    the workload's vocabulary (the shape of the committed loss capture): one untimed log-prob
    pass, `warmup` untimed loss calls, then `steps` timed loss calls and `steps` timed
    log-prob calls with CUDA events.  Prints one JSON line (a kernel measurement, not the
    group-step line)."""
    import torch
    import long_context_grpo_gb300 as ls
    from long_context_grpo_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    torch.cuda.set_device(0)
    R = args.loss_rows
    logits, ids, noise = wl.response_loss_inputs(w, 0, R, args.seed, "cuda")
    old = ls.token_logp(logits, ids) + noise
    loss = torch.zeros(1, dtype=torch.float64, device="cuda")
    dl = torch.empty_like(logits)
    mask = torch.empty((R,), dtype=torch.uint8, device="cuda")
    lp = torch.empty((R,), dtype=torch.float32, device="cuda")
    ws = torch.empty(ls.grpo_loss_workspace_bytes(R), dtype=torch.uint8, device="cuda")
    for _ in range(args.warmup):
        ls.grpo_loss(logits, ids, old, 0.7, w.eps, w.G, loss, dlogits=dl, clip_mask=mask,
                     logp_out=lp, workspace=ws)
    torch.cuda.synchronize()
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    e[0].record()
    for _ in range(args.steps):
        ls.grpo_loss(logits, ids, old, 0.7, w.eps, w.G, loss, dlogits=dl, clip_mask=mask,
                     logp_out=lp, workspace=ws)
    e[1].record()
    for _ in range(args.steps):
        ls.token_logp(logits, ids, logp_out=lp)
    e[2].record()
    torch.cuda.synchronize()
    if ls.device_status() != (0, 0):
        raise RuntimeError("device status set")
    peaks, src = load_peaks()
    ms_l = e[0].elapsed_time(e[1]) / args.steps
    ms_s = e[1].elapsed_time(e[2]) / args.steps
    gb_l = R * (4 * w.V + 12) / (ms_l / 1e3) / 1e9
    gb_s = R * (2 * w.V + 8) / (ms_s / 1e3) / 1e9
    print(json.dumps({"kernel": "grpo_loss + token_logp", "rows": R, "V": w.V,
                      "loss_ms": ms_l, "loss_gbs": gb_l, "loss_frac_hbm": gb_l / peaks["hbm_gbs"],
                      "logp_ms": ms_s, "logp_gbs": gb_s, "logp_frac_hbm": gb_s / peaks["hbm_gbs"],
                      "peak_gbs": peaks["hbm_gbs"], "peak_source": src + " HBM copy"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="p2m")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-rows", type=int, default=8)
    ap.add_argument("--cpu-warmup", type=int, default=1)
    ap.add_argument("--cpu-steps", type=int, default=3)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-score", action="store_true")
    ap.add_argument("--no-packed", action="store_true")
    ap.add_argument("--cp-shards", type=int, default=8,
                    help="prompt shards of the context-parallel measurement (0: skip it)")
    ap.add_argument("--loss-only", action="store_true",
                    help="time only the loss and log-prob kernels on --loss-rows rows")
    ap.add_argument("--loss-rows", type=int, default=4096)
    ap.add_argument("--configs", default="tiny,p32k,p262k,p1m",
                    help="other workloads whose group step is timed too ('' : none)")
    ap.add_argument("--config-steps", type=int, default=2)
    ap.add_argument("--block", type=int, default=4096,
                    help="block length of the blockwise-replay measurement (0: skip it)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("at least 3 warm-up steps")
    from long_context_grpo_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return
        run_reference(args, w)
    elif args.loss_only:
        run_loss_only(args)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()

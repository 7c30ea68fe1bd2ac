#!/usr/bin/env python
"""Benchmark of the speculative-decoding verify step on one GB300 (or N).

A step is one pass of the whole verify path over one batch of the workload:
spec_verify_attn (KV append + masked verify attention, one layer),
spec_reject_sample (temperature softmax, accept/reject, residual/bonus draw)
and kv_commit (rollback / path compaction).  Inputs are seeded synthetic
data resident in HBM before the timed region; the KV cache (GBs) exceeds the
129 MB L2, so no flush is needed between steps.  Each step uses a new
uniform offset so the decisions vary; kv_commit writes the new context
lengths to a separate buffer so every step starts from the same state.

One JSON line on rank 0.  Under torchrun each rank runs its own replica of
the workload (the path shards by request, no collective), timing is the max
over ranks and `value` counts the steps of all ranks ("weak" scaling).

--impl reference times the CPU oracle on the host cores instead, each step a
bounded sample of the same workload (eight requests spread over the context
range) extrapolated to whole steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verify steps/s and accepted tokens/s at 1 GB300; achieved HBM TB/s vs peak"
UNIT = "verify steps/s"
DEFAULT_WORKLOAD = "stress_gqa_152k"
# the two workloads the >= 70%-of-HBM-peak bar is set on
BAR_WORKLOADS = ("stress_gqa_152k", "chain_gqa_128k")

# DRAM traffic of one spec_verify_attn call (request-check/plan kernel and
# the attention kernel with its append and merge) measured by ncu on 16 of
# the 128 requests of the default workload and scaled to 128 by the
# algorithmic bytes (traffic grows with the KV bytes read).  Valid only for
# the attention kernel sources whose digest is recorded with it.
TRAFFIC = {"digest": "fe3f2ab1fed2d51f", "bytes_per_call": 10104592002}
TRAFFIC_ALG_BYTES = 10051956736  # algorithmic bytes per call of that workload (seed 0)


def attn_sources_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_19_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("attn") or f in ("common.cuh", "tc_ptx.cuh"):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def aggregate(ms_local: float, steps: int, world: int, device):
    """Whole-job throughput: the steps of all ranks over the slowest rank's
    time.  Returns (steps_per_s, ms_max)."""
    ms_max = max_over_ranks(ms_local, world, device)
    return world * steps / (ms_max / 1e3), ms_max


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            t0 = time.time()
            while time.time() - t0 < 3.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.02)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 7:
                    continue
                try:
                    sm.append(float(p[0]))
                    smax.append(float(p[1]))
                except ValueError:
                    continue
                for name, v in zip(self.NAMES, p[3:7]):
                    if v.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# the workload
# ---------------------------------------------------------------------------

def build_inputs(wl, seed, device):
    from synth import kv_inputs_device, logits_inputs
    lg = logits_inputs(wl, seed)
    kv = kv_inputs_device(wl, seed, device)
    return lg, kv


def algorithmic_bytes(wl, ctx_lens, parent):
    """Bytes each row of the path must move once (per step)."""
    e = 2 if wl.dtype == "bf16" else 4
    B, M = wl.B, wl.M
    L = ctx_lens.astype(np.int64) + M
    attn = int(L.sum()) * wl.Hkv * wl.D * 2 * e            # K and V read
    attn += B * M * wl.Hkv * wl.D * 2 * e                   # append write
    attn += 2 * B * M * wl.Hq * wl.D * e                    # q read, out write
    if parent is None:
        draft_rows = B * (M - 1)
    else:
        draft_rows = int(sum(len(set(p[1:].tolist())) for p in parent))
    reject = (B * M + draft_rows) * wl.V * e
    return attn, reject


class NativeStep:
    def __init__(self, wl, lg, kv, device, steps_total):
        import speculative_decoding_verification_19_gb300 as sv
        self.sv = sv
        self.wl = wl
        dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        self.dt = dt
        B, M = wl.B, wl.M
        self.dims = sv.make_dims(B=B, M=M, Hq=wl.Hq, Hkv=wl.Hkv, D=wl.D,
                                 max_blocks=kv["max_blocks"], num_blocks=kv["num_blocks"],
                                 V=wl.V, kv_dtype=dt, logits_dtype=dt)
        self.ws = sv.workspace(self.dims, device=device)
        T = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to(device, t)  # noqa: E731
        self.target = T(lg["target"], dt)
        self.draft = T(lg["draft"], dt)
        self.tokens = T(lg["tokens"], torch.int32)
        self.parent = None if lg["parent"] is None else T(lg["parent"], torch.int32)
        self.temperature = T(lg["temperature"], torch.float32)
        self.q, self.k_new, self.v_new = kv["q"], kv["k_new"], kv["v_new"]
        self.k_cache, self.v_cache = kv["k_cache"], kv["v_cache"]
        self.block_table = T(kv["block_table"], torch.int32)
        self.ctx_lens = T(kv["ctx_lens"], torch.int32)
        self.new_ctx = torch.empty_like(self.ctx_lens)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device=device)
        self.out_tokens = torch.empty(B, M, dtype=torch.int32, device=device)
        self.path = torch.empty(B, M, dtype=torch.int32, device=device)
        self.acc = torch.empty(steps_total, B, dtype=torch.int32, device=device)

    def step(self, i, events=None):
        sv = self.sv
        n = 0
        if events:
            events[0].record()
        n += sv.spec_verify_attn(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                 self.block_table, self.ctx_lens, self.parent, self.out,
                                 self.lse, self.dims, self.ws)
        if events:
            events[1].record()
        n += sv.spec_reject_sample(self.target, self.draft, self.tokens, self.parent,
                                   self.temperature, 20261202, i, self.out_tokens, self.path,
                                   self.acc[i], None, self.dims, self.ws)
        if events:
            events[2].record()
        n += sv.kv_commit(self.k_cache, self.v_cache, self.block_table, self.ctx_lens,
                          self.new_ctx, self.path, self.acc[i], self.dims, self.ws)
        if events:
            events[3].record()
        return n

    def host_inputs(self):
        """Pinned host copies of one step's inputs, and pinned result buffers."""
        ins = {k: getattr(self, k).cpu().pin_memory() for k in
               ("q", "k_new", "v_new", "target", "draft", "tokens", "temperature",
                "block_table", "ctx_lens")}
        if self.parent is not None:
            ins["parent"] = self.parent.cpu().pin_memory()
        outs = {"out_tokens": torch.empty_like(self.out_tokens, device="cpu").pin_memory(),
                "path": torch.empty_like(self.path, device="cpu").pin_memory(),
                "acc": torch.empty(self.wl.B, dtype=torch.int32).pin_memory(),
                "new_ctx": torch.empty_like(self.new_ctx, device="cpu").pin_memory()}
        return ins, outs

    def e2e_step(self, i, ins, outs):
        """One step through the public API with this step's inputs copied
        from pinned host memory and its results read back, all inside the
        timed region.  The attention's inputs go first on the compute
        stream; the logits and the decision inputs, which only
        reject-sample reads, come over on two copy streams (in chunks)
        while the attention runs, and reject-sample waits for them.
        Nothing is fetched ahead of its own step."""
        sv = self.sv
        cs = torch.cuda.current_stream()
        if not hasattr(self, "_copy_streams"):
            self._copy_streams = [torch.cuda.Stream() for _ in range(2)]
            self._copy_events = [torch.cuda.Event() for _ in range(2)]
        for k in ("q", "k_new", "v_new", "block_table", "ctx_lens"):
            getattr(self, k).copy_(ins[k], non_blocking=True)
        late = [k for k in ("target", "draft", "tokens", "temperature", "parent") if k in ins]
        for s_, e_ in zip(self._copy_streams, self._copy_events):
            s_.wait_stream(cs)  # the buffers are free once the previous step's work is done
        j = 0
        for k in late:
            dst = getattr(self, k).view(-1)
            src = ins[k].view(-1)
            n = 4 if dst.numel() >= (1 << 20) else 1
            step_ = (dst.numel() + n - 1) // n
            for c in range(n):
                with torch.cuda.stream(self._copy_streams[j % 2]):
                    dst[c * step_:(c + 1) * step_].copy_(src[c * step_:(c + 1) * step_],
                                                       non_blocking=True)
                j += 1
        for s_, e_ in zip(self._copy_streams, self._copy_events):
            e_.record(s_)
        n = sv.spec_verify_attn(self.q, self.k_new, self.v_new, self.k_cache, self.v_cache,
                                self.block_table, self.ctx_lens, self.parent, self.out,
                                self.lse, self.dims, self.ws)
        for e_ in self._copy_events:
            cs.wait_event(e_)
        n += sv.spec_reject_sample(self.target, self.draft, self.tokens, self.parent,
                                   self.temperature, 20261202, i, self.out_tokens, self.path,
                                   self.acc[i], None, self.dims, self.ws)
        n += sv.kv_commit(self.k_cache, self.v_cache, self.block_table, self.ctx_lens,
                          self.new_ctx, self.path, self.acc[i], self.dims, self.ws)
        outs["out_tokens"].copy_(self.out_tokens, non_blocking=True)
        outs["path"].copy_(self.path, non_blocking=True)
        outs["acc"].copy_(self.acc[i], non_blocking=True)
        outs["new_ctx"].copy_(self.new_ctx, non_blocking=True)
        cs.synchronize()
        return n


def timed_steps(st, first, K):
    """K steps bracketed by CUDA events on the launching stream (after a
    synchronize); returns the total and the mean per-call times (ms)."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record()
    for i in range(K):
        st.step(first + i, ev[i])
    t_end.record()
    torch.cuda.synchronize()
    return (t_start.elapsed_time(t_end),
            float(np.mean([e[0].elapsed_time(e[1]) for e in ev])),
            float(np.mean([e[1].elapsed_time(e[2]) for e in ev])),
            float(np.mean([e[2].elapsed_time(e[3]) for e in ev])))


def verify_statistics(wl, acc, st, parent):
    """The pages' observability figures over the timed steps, computed by the
    library's host-side controller: the rejection-position histogram of every
    step (page 2 §5.1), each request's acceptance rate over the steps with
    its histogram and percentiles, and the speculative efficiency (page 3)."""
    from speculative_decoding_verification_19_gb300.controller import Controller, step_stats
    K, B = acc.shape
    pos = np.zeros(wl.M + 1, dtype=np.int64)
    twe = []
    path = st.path.cpu().numpy()  # the last step's path (for the tree figure)
    for k in range(K):
        sst = step_stats(acc[k], path=path if k == K - 1 else None,
                         parent=parent if k == K - 1 else None, M=wl.M)
        pos += np.asarray(sst["rejection_pos"][:wl.M + 1])
        if k == K - 1 and parent is not None:
            twe.append(sst["tree_width_effective"])
    # a controller fed the steps at the workload's fixed draft length (its
    # proposals are reported, not applied: the workload's shape is fixed)
    from speculative_decoding_verification_19_gb300.controller import default_config
    # (a tree's draft length is its depth: the longest path it can accept)
    ctl = Controller(B, gamma0=min(wl.gamma, 63),
                     cfg=default_config(window=min(16, K), max_gamma=63, min_efficiency=0.0))
    proposed = None
    for k in range(K):
        # the draft length stays the workload's: feed each step as drafted at it
        for r in ctl.reqs:
            r.gamma = min(wl.gamma, 63)
        proposed = ctl.update(acc[k])
    m = ctl.metrics()
    out = {"rejection_position_hist": pos.tolist(),
           "acceptance_hist": m["acceptance_hist"],
           "acceptance_p50": round(m["acceptance_p50"], 4),
           "acceptance_p95": round(m["acceptance_p95"], 4),
           "acceptance_p99": round(m["acceptance_p99"], 4),
           "speculative_efficiency": round(m["speculative_efficiency"], 4),
           "proposed_gamma_hist": np.bincount(proposed, minlength=9).tolist()}
    if twe:
        out["tree_width_effective"] = round(float(np.mean(twe)), 4)
    return out


def greedy_reject(st, K, peak, rej_b):
    """spec_reject_sample of the same batch at temperature 0 (greedy:
    exact match with each row's argmax), timed alone on the same inputs."""
    sv = st.sv
    temp0 = torch.zeros_like(st.temperature)
    for i in range(3):
        sv.spec_reject_sample(st.target, st.draft, st.tokens, st.parent, temp0, 1, i,
                              st.out_tokens, st.path, st.acc[0], None, st.dims, st.ws)
    ts = []
    for i in range(K):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record()
        sv.spec_reject_sample(st.target, st.draft, st.tokens, st.parent, temp0, 1, i,
                              st.out_tokens, st.path, st.acc[0], None, st.dims, st.ws)
        b_.record()
        torch.cuda.synchronize()
        ts.append(a_.elapsed_time(b_))
    ms = float(np.mean(ts))
    a = st.acc[0].cpu().numpy()
    assert np.all(a >= 0)
    return {"reject_ms": round(ms, 4), "reject_frac": round(rej_b / (ms / 1e3) / 1e9 / peak, 4),
            "emitted_tokens_per_step": int((a + 1).sum())}


# The LM heads of the stress workload's rows: a 70B-class target (hidden size
# 64 heads x 128) and a small draft head, on random bf16 weights.
LM_HEAD_HT, LM_HEAD_HD = 8192, 1024


def lm_head_step(wl, lg, st, K, peaks):
    """spec_reject_sample_lm_head on the default workload's shape (the
    statistics formed in the LM heads' epilogue) against the same LM heads
    followed by spec_reject_sample (a second pass over the logit rows),
    each timed over K calls with CUDA events; the target head alone gives the
    tensor-core rate."""
    sv = st.sv
    dev = st.target.device
    B, M, V = wl.B, wl.M, wl.V
    g = torch.Generator(device=dev)
    g.manual_seed(20261202)
    ht = torch.randn(B, M, LM_HEAD_HT, device=dev, generator=g).to(torch.bfloat16)
    wt = (torch.randn(V, LM_HEAD_HT, device=dev, generator=g) * (3.0 / LM_HEAD_HT ** 0.5)).to(torch.bfloat16)
    hd = torch.randn(B, M, LM_HEAD_HD, device=dev, generator=g).to(torch.bfloat16)
    wd = (torch.randn(V, LM_HEAD_HD, device=dev, generator=g) * (3.0 / LM_HEAD_HD ** 0.5)).to(torch.bfloat16)
    tl = torch.empty(B, M, V, dtype=torch.bfloat16, device=dev)
    dl = torch.empty_like(tl)
    ws = st.ws

    def fused(i):
        return sv.spec_reject_sample_lm_head(ht, wt, hd, wd, tl, dl, st.tokens, st.parent,
                                             st.temperature, 3, i, st.out_tokens, st.path,
                                             st.acc[0], None, st.dims, ws)

    def unfused(i):
        n = sv.spec_lm_head(ht.view(B * M, -1), wt, tl.view(B * M, -1), ws)
        n += sv.spec_lm_head(hd.view(B * M, -1), wd, dl.view(B * M, -1), ws)
        n += sv.spec_reject_sample(tl, dl, st.tokens, st.parent, st.temperature, 3, i,
                                   st.out_tokens, st.path, st.acc[0], None, st.dims, ws)
        return n

    def target_head(i):
        return sv.spec_lm_head(ht.view(B * M, -1), wt, tl.view(B * M, -1), ws)

    res = {}
    for name, f in (("fused", fused), ("unfused", unfused), ("target_head", target_head)):
        for i in range(3):
            f(i)
        torch.cuda.synchronize()
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record()
        for i in range(K):
            launches = f(i)
        b_.record()
        torch.cuda.synchronize()
        res[name] = (a_.elapsed_time(b_) / K, launches)
    assert sv.device_status(ws) == 0
    a = st.acc[0].cpu().numpy()
    assert np.all(a >= 0)
    flops = 2.0 * B * M * LM_HEAD_HT * V
    t_ms = res["target_head"][0]
    achieved = flops / (t_ms / 1e3) / 1e12
    return {"workload": f"{wl.name} rows (B {B} x M {M}), V {V}, target hidden {LM_HEAD_HT}, "
                        f"draft hidden {LM_HEAD_HD}, random bf16 weights",
            "fused_ms": round(res["fused"][0], 4), "fused_launches": res["fused"][1],
            "unfused_ms": round(res["unfused"][0], 4), "unfused_launches": res["unfused"][1],
            "target_head_ms": round(t_ms, 4),
            "roofline": {"bound": "tensor", "kernel": "lm_head_kernel (target head)",
                         "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                         "peak_source": peaks["source"] + " bf16 burst", "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "flops_per_call": flops}}


def run_only(args, wl):
    """One entry point alone on the workload's shapes: W untimed calls, then
    K calls between CUDA events (no flush: for profiler captures and per-call
    comparisons, not a bench line).  reject: spec_reject_sample on the
    workload's logits; lm_head: spec_lm_head on rows B x M of random hidden
    states against a random V x LM_HEAD_HT weight."""
    import speculative_decoding_verification_19_gb300 as sv
    from synth import logits_inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    B, M, V = wl.B, wl.M, wl.V
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    T = lambda x, t: torch.from_numpy(np.ascontiguousarray(x)).to(dev, t)  # noqa: E731
    if args.only == "reject":
        lg = logits_inputs(wl, args.seed)
        dims = sv.make_dims(B=B, M=M, V=V, logits_dtype=dt)
        ws = sv.workspace(dims, device=dev)
        tgt, dft = T(lg["target"], dt), T(lg["draft"], dt)
        tok, temp = T(lg["tokens"], torch.int32), T(lg["temperature"], torch.float32)
        par = None if lg["parent"] is None else T(lg["parent"], torch.int32)
        out = torch.empty(B, M, dtype=torch.int32, device=dev)
        path = torch.empty_like(out)
        acc = torch.empty(B, dtype=torch.int32, device=dev)

        def call(i):
            return sv.spec_reject_sample(tgt, dft, tok, par, temp, 20261202, i, out, path, acc,
                                         None, dims, ws)
    else:
        g = torch.Generator(device=dev)
        g.manual_seed(20261202)
        h = torch.randn(B * M, LM_HEAD_HT, device=dev, generator=g).to(torch.bfloat16)
        w = (torch.randn(V, LM_HEAD_HT, device=dev, generator=g)
             * (3.0 / LM_HEAD_HT ** 0.5)).to(torch.bfloat16)
        logits = torch.empty(B * M, V, dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(64, dtype=torch.uint8, device=dev)

        def call(i):
            return sv.spec_lm_head(h, w, logits, ws)
    for i in range(args.warmup):
        call(i)
    torch.cuda.synchronize()
    a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_.record()
    for i in range(args.steps):
        launches = call(args.warmup + i)
    b_.record()
    torch.cuda.synchronize()
    assert sv.device_status(ws) == 0
    ms = a_.elapsed_time(b_) / args.steps
    line = {"only": args.only, "workload": wl.name, "B": B, "M": M, "V": V,
            "ms_per_call": round(ms, 4), "launches_per_call": launches, "calls": args.steps}
    if args.only == "lm_head":
        line["tflops"] = round(2.0 * B * M * LM_HEAD_HT * V / (ms / 1e3) / 1e12, 1)
    print(json.dumps(line), flush=True)


def second_workload(name, seed, device, K, W, peak):
    """The other workload the HBM bar is set on, timed the same way in the
    same process after the main timed region (its own inputs, K steps)."""
    from synth import workload
    wl = workload(name)
    lg, kv = build_inputs(wl, seed, device)
    st = NativeStep(wl, lg, kv, device, W + 1 + K)
    attn_b, rej_b = algorithmic_bytes(wl, kv["ctx_lens"], lg["parent"])
    for i in range(W + 1):
        st.step(i)
    ms_total, attn_ms, rej_ms, com_ms = timed_steps(st, W + 1, K)
    acc = st.acc[W + 1:W + 1 + K].cpu().numpy()
    assert np.all(acc >= 0), "a request failed inside the timed region"
    res = {"steps_per_s": round(K / (ms_total / 1e3), 3),
           "ms_per_step": round(ms_total / K, 4),
           "attn_ms": round(attn_ms, 4), "reject_ms": round(rej_ms, 4),
           "commit_ms": round(com_ms, 4),
           "attn_bytes": attn_b, "reject_bytes": rej_b,
           "attn_frac": round(attn_b / (attn_ms / 1e3) / 1e9 / peak, 4),
           "reject_frac": round(rej_b / (rej_ms / 1e3) / 1e9 / peak, 4),
           "emitted_tokens_per_step": round(float((acc + 1).sum(axis=1).mean()), 2),
           "config": {"B": wl.B, "gamma": wl.gamma, "M": wl.M, "V": wl.V, "Hq": wl.Hq,
                      "Hkv": wl.Hkv, "D": wl.D, "ctx": list(wl.ctx)}}
    del st, lg, kv
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample
# ---------------------------------------------------------------------------

class OracleSample:
    """The oracle over single requests of the workload (host copies)."""

    def __init__(self, wl, lg, kv, reqs):
        self.wl = wl
        self.lg = lg
        self.reqs = list(reqs)
        self.data = {}
        bt = kv["block_table"]
        for b in self.reqs:
            pages = bt[b][bt[b] >= 0]
            idx = torch.from_numpy(pages.astype(np.int64)).to(kv["k_cache"].device)
            kc = kv["k_cache"].index_select(0, idx).float().cpu().numpy()
            vc = kv["v_cache"].index_select(0, idx).float().cpu().numpy()
            table = np.arange(len(pages), dtype=np.int32)[None]
            self.data[b] = dict(
                kc=kc, vc=vc, table=table, ctx=kv["ctx_lens"][b:b + 1],
                q=kv["q"][b:b + 1].float().cpu().numpy(),
                kn=kv["k_new"][b:b + 1].float().cpu().numpy(),
                vn=kv["v_new"][b:b + 1].float().cpu().numpy())

    def run(self, b, offset):
        from oracle import oracle_kv_commit, oracle_reject_sample, oracle_verify_attn
        d = self.data[b]
        par = None if self.lg["parent"] is None else self.lg["parent"][b:b + 1]
        _, _, kc, vc = oracle_verify_attn(d["q"], d["kc"], d["vc"], d["table"], d["ctx"],
                                          d["kn"], d["vn"], parent=par)
        r = oracle_reject_sample(self.lg["target"][b:b + 1], self.lg["draft"][b:b + 1],
                                 self.lg["tokens"][b:b + 1], par,
                                 self.lg["temperature"][b:b + 1], 20261202, offset,
                                 b_base=b)
        oracle_kv_commit(kc, vc, d["table"], d["ctx"], r["path"], r["accepted_len"])
        return r


def sample_requests(ctx_lens, n=8):
    """n requests spread over the context range: the ones at evenly spaced
    ranks of the context lengths (shortest and longest included)."""
    order = np.argsort(np.asarray(ctx_lens), kind="stable")
    n = min(n, len(order))
    ranks = np.unique(np.round(np.linspace(0, len(order) - 1, n)).astype(int))
    return [int(order[r]) for r in ranks]


def cpu_baseline(wl, lg, kv):
    """The oracle on the sampled requests of one step, scaled to whole steps."""
    reqs = sample_requests(kv["ctx_lens"])
    sample = OracleSample(wl, lg, kv, reqs)
    t0 = time.perf_counter()
    for b in reqs:
        sample.run(b, 0)
    el = time.perf_counter() - t0
    return {"value": (len(reqs) / wl.B) / el, "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle", "requests": reqs,
            "sample": f"requests {reqs} of the {wl.B} of one step (spread over the context "
                      f"range), each through the fp64 numpy oracle: append+attention over all "
                      f"{wl.Hkv} KV heads, reject-sample, commit; {el:.1f} s; value "
                      f"extrapolated to whole steps as {len(reqs)}/{wl.B} of a step"}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_native(args, wl, world, rank, local):
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist_init(world, "nccl")
    seed = args.seed + rank
    lg, kv = build_inputs(wl, seed, device)
    K, W = args.steps, args.warmup
    st = NativeStep(wl, lg, kv, device, max(K, W, 1) + W + K)
    attn_b, rej_b = algorithmic_bytes(wl, kv["ctx_lens"], lg["parent"])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, lg, kv)

    for i in range(W):
        st.step(i)
    torch.cuda.synchronize()
    launches_per_step = st.step(W)  # one more untimed step to count launches
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    ms_total, attn_ms, rej_ms, com_ms = timed_steps(st, W + 1, K)
    barrier(world)
    clk = clocks.stop()
    steps_per_s, ms_max = aggregate(ms_total, K, world, device)
    acc = st.acc[W + 1:W + 1 + K].cpu().numpy()
    assert np.all(acc >= 0), "a request failed inside the timed region"
    emitted_per_step = float((acc + 1).sum(axis=1).mean())
    verify_stats = verify_statistics(wl, acc, st, lg["parent"])

    # end to end through the public API with pinned host buffers
    ins, outs = st.host_inputs()
    h2d = sum(v.numel() * v.element_size() for v in ins.values())
    d2h = sum(v.numel() * v.element_size() for v in outs.values())
    for i in range(2):
        st.e2e_step(i, ins, outs)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(K):
        st.e2e_step(i, ins, outs)
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, device)

    peaks = measured_peaks()
    # both workloads the HBM bar is set on, in the same line: this one from
    # the timed region above, the other timed after it in this process
    workloads = {wl.name: {"attn_frac": round(attn_b / (attn_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                           "reject_frac": round(rej_b / (rej_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4)}}
    workloads[wl.name + " (temperature 0)"] = greedy_reject(st, K, peaks["hbm_gbs"], rej_b)
    lm_head = lm_head_step(wl, lg, st, K, peaks) if not args.no_second else None
    if not args.no_second and wl.name in BAR_WORKLOADS:
        for other in BAR_WORKLOADS:
            if other != wl.name:
                workloads[other] = second_workload(other, seed, device, K, W, peaks["hbm_gbs"])
    achieved = attn_b / (attn_ms / 1e3) / 1e9
    # the recorded traffic belongs to the default workload at its full size
    # (the bytes per call of the run it was scaled to) and to these sources
    traffic = (TRAFFIC["bytes_per_call"]
               if TRAFFIC["digest"] == attn_sources_digest() and attn_b == TRAFFIC_ALG_BYTES
               else None)
    line = {
        "metric": METRIC, "value": round(steps_per_s, 3), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_max / K, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "gamma": wl.gamma, "M": wl.M,
                   "V": wl.V, "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D,
                   "ctx": list(wl.ctx), "layers": 1,
                   "parallelism": f"replicas x{world} (request shards, no collective)",
                   "l2": "inputs larger than L2 (KV cache %.1f GB), no flush"
                         % (2 * kv["k_cache"].numel() * kv["k_cache"].element_size() / 1e9)},
        "accepted_tokens_per_s": round(steps_per_s * emitted_per_step, 1),
        "emitted_tokens_per_step": round(emitted_per_step, 2),
        "hbm_tb_s": round((attn_b + rej_b) / (ms_max / K / 1e3) / 1e12, 3),
        "roofline": {"bound": "hbm", "kernel": "spec_verify_attn (request checks + plan, attention with append and merge)",
                     "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                     "peak_source": peaks["source"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "bytes_per_call": attn_b, "traffic": traffic},
        "kernels": {"attn_ms": round(attn_ms, 4), "reject_ms": round(rej_ms, 4),
                    "commit_ms": round(com_ms, 4),
                    "reject_gbs": round(rej_b / (rej_ms / 1e3) / 1e9, 1),
                    "reject_frac": round(rej_b / (rej_ms / 1e3) / 1e9 / peaks["hbm_gbs"], 4),
                    "reject_bytes": rej_b},
        "workloads": workloads,
        "lm_head": lm_head,
        "verify_stats": verify_stats,
        "cpu_baseline": cpu,
        "e2e": {"value": round(world * K / e2e_s, 3), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * K,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args, wl, world, rank):
    if rank != 0:
        return
    from synth import context_lengths, kv_inputs_host, logits_inputs
    lg = logits_inputs(wl, args.seed)
    K, W = args.steps, args.warmup
    ctx_all = context_lengths(wl, args.seed)
    reqs = sample_requests(ctx_all)   # the same requests the native arm's baseline times
    n = len(reqs)
    # host-side inputs of those requests only (their own pages, same lengths)
    kv = kv_inputs_host(wl.scaled(B=n), args.seed, ctx=ctx_all[reqs])
    kvt = dict(kv)
    for k in ("q", "k_new", "v_new", "k_cache", "v_cache"):
        kvt[k] = torch.from_numpy(kv[k])
    sub = {k: (v[reqs] if isinstance(v, np.ndarray) and v.shape[:1] == (wl.B,) else v)
           for k, v in lg.items()}
    sample = OracleSample(wl, sub, kvt, range(n))
    # a warm-up step is one request; each timed step runs every sampled request
    for i in range(W):
        sample.run(i % n, i)
    t0 = time.perf_counter()
    for i in range(K):
        for j in range(n):
            sample.run(j, W + i)
    el = time.perf_counter() - t0
    value = (K * n / wl.B) / el
    # a step of this arm is the sampled one (n of the B requests): its time
    # is what the clock saw; the value is extrapolated to whole steps
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT,
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": round(1e3 * el / K, 1),
        "ms_per_whole_step_extrapolated": round(1e3 / value, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "gamma": wl.gamma, "V": wl.V,
                   "Hq": wl.Hq, "Hkv": wl.Hkv, "D": wl.D, "ctx": list(wl.ctx)},
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": os.cpu_count(),
                         "kind": "oracle", "requests": reqs,
                         "sample": f"each timed step = requests {reqs} of the {wl.B} "
                                   "(spread over the context range) through the fp64 numpy "
                                   "oracle (append+attention, reject-sample, commit); "
                                   "ms_per_step is that sampled step's time, the value "
                                   f"extrapolated to whole steps as {n}/{wl.B} of a step"},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--batch", type=int, default=None,
                    help="requests per step (default: the workload's batch)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-second", action="store_true",
                    help="time only the selected workload")
    ap.add_argument("--only", choices=("reject", "lm_head"), default=None,
                    help="run one entry point alone (for profiler captures); no bench line")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # at least three untimed steps
    from synth import workload
    wl = workload(args.workload)
    if args.batch is not None:
        wl = wl.scaled(B=args.batch)
    if args.only is not None:
        run_only(args, wl)
        return
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, wl, world, rank)
    else:
        run_native(args, wl, world, rank, local)


if __name__ == "__main__":
    main()

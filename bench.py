#!/usr/bin/env python
"""Benchmark of the SSE layer hot path on GB300: tokens/s (forward + decode).

One step = one sse_forward over the 2B-scale layer batch (8 sequences x 4096
tokens, 16 heads, c = d = 128, N = 8, top-2, shared partition; bf16 token
tensors, fp32 states) followed by one sse_decode_step over the decode batch
(256 sequences x 16 heads, c = d = 128, N = 16, top-2, shared; fp32 states
resident in HBM).  value = tokens processed per second over both calls
(32768 + 256 tokens per step), with inputs resident in HBM; every forward and
decode input is larger than the 129 MB L2 (545 MB of token tensors, 4.6 GB
of decode states), so no L2 flush is needed between steps.

Also reported: per-kernel CUDA-event timing of the dominant kernel against
the measured HBM peak (roofline), the end-to-end number through the C ABI
with host buffers (pinned host -> device copies of every step's inputs and
device -> host copies of its outputs inside the timed region, on copy streams
that overlap one step's transfers with the neighbouring steps' compute), SM clocks
sampled during the timed region, and the fp64 CPU oracle timed on a bounded
sample of the same workload (cpu_baseline).

``--impl reference`` times the CPU oracle alone on bounded samples of the same
workload (the reference arm: the pages publish no code to run).
Multi-GPU (torchrun): every rank runs its own batch (weak scaling, no
collective on the data path); rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from sparse_state_linear_router_gb300 import inputs as synth  # noqa: E402

METRIC = "SSE layer tokens/s (fwd + decode) on 1 GB300; % of binding HBM/tensor roofline"
FWD_WORKLOAD = "layer_bf16"
DEC_WORKLOAD = "decode_bf16"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def profiled_traffic(kernel: str):
    """DRAM bytes (read + write) per launch of a kernel from the ncu capture
    recorded in profiles/dram_traffic.json, or None once the kernel's source
    no longer has the hash recorded there (the counters then describe another
    build).  Returns (bytes, the summary that documents the capture)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            entry = json.load(f)[kernel]
        with open(os.path.join(ROOT, entry["source"]), "rb") as f:
            digest = hashlib.sha256(f.read()).hexdigest()
    except (OSError, KeyError, ValueError):
        return None, None
    if entry.get("source_sha256") != digest:
        return None, None
    return int(entry["dram_bytes_per_launch"]), entry.get("summary")


# ---------------------------------------------------------------------------
# Algorithmic work (compulsory bytes: inputs read once, outputs written once;
# flops of the recurrence: 4cd per token, head and active partition)
# ---------------------------------------------------------------------------
def _sz(w):
    return 2 if w.dtype == "bf16" else 4


def forward_main_bytes(w, T, S, init=False, final=True):
    s = _sz(w)
    H, c, d, P = w.num_heads, w.key_dim, w.value_dim, w.num_slots
    b = T * H * (3 * c + d) * s + T * H * d * s
    st = S * H * P * c * d * 4
    return b + (st if final else 0) + (st if init else 0)


def forward_step_bytes(w, T, S, init=False, final=True):
    return forward_main_bytes(w, T, S, init, final) + T * w.num_heads * w.num_partitions * _sz(w)


def forward_flops(w, T):
    a = w.top_k + w.use_shared
    return T * w.num_heads * a * 4 * w.key_dim * w.value_dim


def decode_bytes(w, B):
    s = _sz(w)
    H, c, d, N = w.num_heads, w.key_dim, w.value_dim, w.num_partitions
    a = w.top_k + w.use_shared
    return B * H * (a * c * d * 4 * 2 + (3 * c + d + N) * s + d * s)


def decode_flops(w, B):
    return B * w.num_heads * (w.top_k + w.use_shared) * 4 * w.key_dim * w.value_dim


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "25"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.out or "")) if len(r) >= 10]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}

        def num(x):
            try:
                return float(x.strip())
            except ValueError:
                return None
        busy = [r for r in rows if (num(r[4]) or 0) >= 50] or rows
        sm = [num(r[1]) for r in busy if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i in range(4) if r[6 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": num(busy[0][2]), "reasons": reasons, "samples": len(busy),
                "power_w_max": max((num(r[3]) or 0) for r in busy)}


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample (cpu_baseline / reference arm)
# ---------------------------------------------------------------------------
class OracleSampler:
    """Times the fp64 CPU oracle on bounded samples of the workload: the
    forward over sequence 0 of the forward batch (all heads) and one decode
    step over the first ``dec_seqs`` decode sequences (all heads)."""

    def __init__(self, fwd_inp, w_fwd, dec_steps, w_dec, dec_seqs=16):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.w_fwd, self.w_dec, self.dec_seqs = w_fwd, w_dec, dec_seqs
        t0, t1 = int(fwd_inp.cu_seqlens[0]), int(fwd_inp.cu_seqlens[1])
        self.fwd_tokens = t1 - t0
        self.sub = {n: np.ascontiguousarray(getattr(fwd_inp, n)[t0:t1]) for n in ("q", "k", "v", "g", "logits")}
        self.cu = np.array([0, t1 - t0], dtype=np.int64)
        self.dec = [{n: np.ascontiguousarray(getattr(x, n)[:dec_seqs]) for n in ("q", "k", "v", "g", "logits")}
                    for x in dec_steps]
        self.state = np.zeros((dec_seqs, w_dec.num_heads, w_dec.num_slots, w_dec.key_dim, w_dec.value_dim))
        self.fwd_time = self.dec_time = 0.0
        self.fwd_n = self.dec_n = 0
        self.threads = 1
        self.iters = 0

    def once(self):
        w, s = self.w_fwd, self.sub
        a = time.perf_counter()
        r = self.oracle.forward(s["q"], s["k"], s["v"], s["g"], s["logits"], self.cu, top_k=w.top_k,
                                use_shared=w.use_shared)
        self.fwd_time += time.perf_counter() - a
        self.fwd_n += self.fwd_tokens
        self.threads = max(self.threads, r["threads"])
        x = self.dec[self.iters % len(self.dec)]
        a = time.perf_counter()
        r = self.oracle.decode_step(self.state, x["q"], x["k"], x["v"], x["g"], x["logits"],
                                    top_k=self.w_dec.top_k, use_shared=self.w_dec.use_shared)
        self.dec_time += time.perf_counter() - a
        self.dec_n += self.dec_seqs
        self.threads = max(self.threads, r["threads"])
        self.iters += 1

    def run_for(self, seconds):
        start = time.perf_counter()
        while self.iters == 0 or time.perf_counter() - start < seconds:
            self.once()

    def reset(self):
        self.fwd_time = self.dec_time = 0.0
        self.fwd_n = self.dec_n = 0
        self.iters = 0

    def rates(self):
        return self.fwd_n / self.fwd_time, self.dec_n / self.dec_time

    def sample_text(self):
        return (f"forward: sequence 0 of the forward batch ({self.fwd_tokens} tokens x {self.w_fwd.num_heads} "
                f"heads); decode: {self.dec_seqs} of {self.w_dec.decode_batch} sequences x "
                f"{self.w_dec.num_heads} heads, one step; {self.iters} repetitions")


def step_equivalent_tps(fwd_tokens, dec_tokens, fwd_tps, dec_tps):
    """Tokens/s of one full step (forward batch + decode batch) at the given rates."""
    return (fwd_tokens + dec_tokens) / (fwd_tokens / fwd_tps + dec_tokens / dec_tps)


# ---------------------------------------------------------------------------
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_barrier(ws):
    """Barrier over all ranks of the job (no-op for one process)."""
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks_of(x, ws, dev):
    """Largest value of the scalar x over all ranks (the slowest rank's time)."""
    if ws > 1:
        import torch
        import torch.distributed as dist
        tt = torch.tensor([float(x)], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        return float(tt.item())
    return x


def whole_job_tokens_per_s(ws, tokens_per_rank_step, ms_per_step):
    """Weak scaling: every rank processes its own batch of tokens_per_rank_step
    tokens per step; the job rate is all ranks' tokens over the slowest rank's
    step time."""
    return ws * tokens_per_rank_step / (ms_per_step * 1e-3)


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    w_fwd, w_dec = synth.WORKLOADS[args.fwd_workload], synth.WORKLOADS[DEC_WORKLOAD]
    if args.decode_batch:  # a smaller decode batch (profiling captures)
        import dataclasses
        w_dec = dataclasses.replace(w_dec, decode_batch=args.decode_batch)
    fwd_inp = synth.make_forward_inputs(w_fwd, seed=0)
    dec_steps = [synth.make_decode_inputs(w_dec, s, batch=16) for s in range(4)]
    T = fwd_inp.total_tokens
    B = w_dec.decode_batch
    do_fwd = args.part in ("both", "forward")
    do_dec = args.part in ("both", "decode")
    smp = OracleSampler(fwd_inp, w_fwd, dec_steps, w_dec, dec_seqs=16)
    for _ in range(args.warmup):
        smp.once()
    smp.reset()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.once()
    wall = time.perf_counter() - t0
    fwd_tps, dec_tps = smp.rates()
    if do_fwd and do_dec:
        value = step_equivalent_tps(T, B, fwd_tps, dec_tps)
    else:
        value = fwd_tps if do_fwd else dec_tps
    parts = ([describe_forward(w_fwd, fwd_inp)] if do_fwd else []) + ([describe_decode(w_dec)] if do_dec else [])
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": " + ".join(parts), "fwd_tokens_per_step": T if do_fwd else 0,
                   "decode_tokens_per_step": B if do_dec else 0},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": smp.threads, "kind": "oracle",
                         "sample": "per step: " + smp.sample_text() + "; value = tokens/s of one full step "
                                                                       "at the measured forward and decode rates"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def describe_forward(w, inp):
    lens = np.diff(inp.cu_seqlens)
    shape = (f"{inp.num_seqs} seqs x {int(lens[0])} tokens" if np.all(lens == lens[0])
             else f"{inp.num_seqs} varlen seqs, {inp.total_tokens} tokens")
    return (f"{w.name} forward ({shape}, H{w.num_heads}, c={w.key_dim}, d={w.value_dim}, "
            f"N{w.num_partitions}, top-{w.top_k}{', shared' if w.use_shared else ''}, {w.dtype} in, fp32 state"
            f"{', random initial state' if inp.init_state is not None else ''})")


def describe_decode(w):
    return (f"{w.name} step ({w.decode_batch} seqs x H{w.num_heads}, c={w.key_dim}, d={w.value_dim}, "
            f"N{w.num_partitions}, top-{w.top_k}{', shared' if w.use_shared else ''}, fp32 states resident)")


def graph_replay_ms(call, reps=50):
    """Mean time of one replay of a CUDA graph holding call(stream) (captured
    after two warm-up calls on a side stream), CUDA events around `reps`
    back-to-back replays."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            call(side.cuda_stream)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(torch.cuda.current_stream().cuda_stream)
    g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    del g
    return e0.elapsed_time(e1) / reps


def time_forward_variants(args, dev, peaks):
    """Forward-only timings of the other forward workloads, reported beside
    the step (not part of `value`): the long-context varlen batch (16
    sequences, lengths U[1024, 32768] with the seed-0 draw, H16, N16, random
    initial state, initial and final state I/O), the small batch (B2 T2048 H4
    c=d=64 N8) under both schedules, and the layer batch with a per-partition
    router bias that skews the partition loads (stress variant) under both
    schedules.  Inputs are drawn on the device (same distributions as the
    parity tests' numpy generator, another stream of numbers); each is larger
    than L2 except the small batch (4 MB), whose time is launch-bound."""
    import torch
    from sparse_state_linear_router_gb300 import binding
    stream = torch.cuda.current_stream(dev)
    hbm, tflops = peaks["hbm_gbs"], peaks["bf16_tflops"]
    P_ = binding._ptr
    res = {}
    N8 = synth.WORKLOADS["layer_bf16"].num_partitions
    skew = 1.5 * (np.arange(N8) / (N8 - 1) - 0.5) * 2.0
    import dataclasses
    k_eq_n = dataclasses.replace(synth.WORKLOADS["small_bf16"], name="small_bf16_k4_of_4", num_partitions=4,
                                 top_k=4)
    cases = [("varlen_bf16", "varlen_bf16", None, "auto"),
             ("small_bf16", "small_bf16", None, "auto"),
             ("small_bf16_masked", "small_bf16", None, "masked"),
             ("small_bf16_k4_of_4", k_eq_n, None, "auto"),
             ("small_bf16_k4_of_4_grouped", k_eq_n, None, "chunked"),
             ("layer_bf16_skewed", "layer_bf16", skew, "auto"),
             ("layer_bf16_skewed_masked", "layer_bf16", skew, "masked")]
    for key, wname, bias, algo in cases:
        w = synth.WORKLOADS[wname] if isinstance(wname, str) else wname
        x = synth.make_forward_inputs_device(w, seed=0, device=dev, router_bias=bias)
        T, S = x["total_tokens"], x["num_seqs"]
        cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, w.top_k,
                                  w.use_shared, 1.0, w.dtype, algo)
        out = torch.empty((T, w.num_heads, w.value_dim), dtype=torch.bfloat16, device=dev)
        fin = torch.empty((S, w.num_heads, w.num_slots, w.key_dim, w.value_dim), dtype=torch.float32, device=dev)
        wsp = binding.forward_workspace(cfg, T, S, dev)
        nl = {"n": 0}

        def call(evs=None):
            st, n = binding.sse_forward_timed(cfg, P_(x["q"]), P_(x["k"]), P_(x["v"]), P_(x["g"]),
                                              P_(x["logits"]), None, None, P_(x["cu_seqlens"]), S, T,
                                              P_(x["init"]), P_(fin), P_(out), None, None, P_(wsp), wsp.numel(),
                                              stream.cuda_stream,
                                              None if evs is None else [e.cuda_event for e in evs])
            binding._check(st, "sse_forward_timed")
            nl["n"] = n
        for _ in range(max(3, args.warmup)):
            call()
        reps = 10
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
        for e4 in evs:
            for e in e4:
                e.record(stream)
        torch.cuda.synchronize()
        for i in range(reps):
            call(evs[i])
        torch.cuda.synchronize()
        st, flags = binding.sse_read_device_status(wsp.data_ptr(), stream.cuda_stream)
        ms = statistics.mean(e[0].elapsed_time(e[3]) for e in evs)
        main_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
        has_init = x["init"] is not None
        fb = forward_step_bytes(w, T, S, init=has_init)
        ff = forward_flops(w, T)
        t_bind = max(ff / (tflops * 1e12), fb / (hbm * 1e9))
        mb = forward_main_bytes(w, T, S, init=has_init)
        res[key] = {
            "workload": describe_forward(w, synth.LayerInputs(w, None, None, None, None, None,
                                                              x["cu_seqlens"].cpu().numpy(),
                                                              np.zeros(1) if has_init else None)),
            "algo": algo, "router_bias": None if bias is None else [round(float(b), 4) for b in bias],
            "ms": ms, "route_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in evs),
            "main_ms": main_ms, "tail_ms": statistics.mean(e[2].elapsed_time(e[3]) for e in evs),
            "tokens_per_s": T / (ms * 1e-3), "launches": nl["n"],
            "roofline": {"bound": "hbm" if fb / (hbm * 1e9) >= ff / (tflops * 1e12) else "tensor",
                         "binding_ms": t_bind * 1e3, "frac": t_bind / (ms * 1e-3),
                         "main_kernel_gbs": mb / (main_ms * 1e6), "main_kernel_frac_of_hbm": mb / (main_ms * 1e6) / hbm,
                         "algorithmic_bytes": fb, "algorithmic_flops": ff},
            "device_status": st, "device_flags": flags,
        }
        if wname == "small_bf16" and bias is None:
            # the launch-bound shape replayed as one CUDA graph of the same call
            g_ms = graph_replay_ms(lambda s: binding._check(
                binding.sse_forward(cfg, P_(x["q"]), P_(x["k"]), P_(x["v"]), P_(x["g"]), P_(x["logits"]), None,
                                    None, P_(x["cu_seqlens"]), S, T, P_(x["init"]), P_(fin), P_(out), None, None,
                                    P_(wsp), wsp.numel(), s), "sse_forward"))
            res[key]["graph_ms"] = g_ms
            res[key]["graph_tokens_per_s"] = T / (g_ms * 1e-3)
        del x, out, fin, wsp
        torch.cuda.empty_cache()
    return res


def time_fwd_bwd_fig6(args, dev, L=8192):
    """Forward and backward times at the operator shape of the pages' Fig. 6
    ("Scaling Linear Attention with Sparse State Expansion", section 2.6:
    8 heads, head dim 128, top-1, N = 4 / 8 / 16, cu_seqlens = [0, L/2, L]),
    bf16 token tensors, fp32 states, d_out ~ N(0, 1); the pages give no
    numbers for it (a figure only)."""
    import dataclasses

    import torch
    from sparse_state_linear_router_gb300 import binding
    stream = torch.cuda.current_stream(dev)
    P_ = binding._ptr
    res = {}
    for N in (4, 8, 16):
        w = dataclasses.replace(synth.WORKLOADS["layer_bf16"], name=f"fig6_N{N}", num_heads=8, num_partitions=N,
                                top_k=1, lengths=(L // 2, L // 2), sigma_router=1.0)
        x = synth.make_forward_inputs_device(w, seed=0, device=dev)
        T, S = x["total_tokens"], x["num_seqs"]
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        d_out = torch.randn((T, w.num_heads, w.value_dim), generator=gen, device=dev).to(torch.bfloat16)
        cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, N, 1, 1, 1.0, "bf16")
        fws = binding.forward_workspace(cfg, T, S, dev)
        bws = torch.empty(binding.sse_backward_workspace_size(cfg, T, S), dtype=torch.uint8, device=dev)
        out = torch.empty((T, w.num_heads, w.value_dim), dtype=torch.bfloat16, device=dev)

        def fwd():
            binding.forward(cfg, x["q"], x["k"], x["v"], x["g"], x["logits"], x["cu_seqlens"], out=out,
                            want_final_state=False, workspace=fws)

        def bwd():
            binding.backward(cfg, x["q"], x["k"], x["v"], x["g"], x["logits"], x["cu_seqlens"], d_out,
                             want_d_initial_state=False, workspace=bws)

        times = {}
        for name, fn, reps in (("forward", fwd, 10), ("backward", bwd, 3)):
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            times[name + "_ms"] = e0.elapsed_time(e1) / reps
        res[f"N{N}"] = dict(times, fwd_bwd_ms=times["forward_ms"] + times["backward_ms"],
                            workload=f"H8, c=d=128, top-1 of N={N}, shared, cu_seqlens=[0, {L // 2}, {L}], bf16")
        del x, fws, bws, out, d_out
        torch.cuda.empty_cache()
    return res


def delta_inputs(w, T, dev, seed=None, gen=None):
    """One batch of T tokens for the delta rule, drawn on the device: unit
    keys, q = N(0,1)/sqrt(c), v = N(0,1), log_alpha = logsigmoid(N(0,1))/16
    and beta = sigmoid(N(0,1)) per (token, head), router logits N(0, sigma_r);
    bf16.  `gen` (a torch generator) continues a stream; else one is seeded."""
    import torch
    if gen is None:
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed)

    def normal(*shape):
        return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32)
    H, c, d, N = w.num_heads, w.key_dim, w.value_dim, w.num_partitions
    k = normal(T, H, c)
    return {"q": (normal(T, H, c) / np.sqrt(c)).to(torch.bfloat16),
            "k": (k / k.norm(dim=-1, keepdim=True)).to(torch.bfloat16),
            "v": normal(T, H, d).to(torch.bfloat16),
            "la": (torch.nn.functional.logsigmoid(normal(T, H)) / 16).to(torch.bfloat16),
            "b": torch.sigmoid(normal(T, H)).to(torch.bfloat16),
            "lg": (normal(T, H, N) * w.sigma_router).to(torch.bfloat16)}


def time_delta(args, dev):
    """SSE on the gated delta rule (CUDA cores): the forward on the layer
    workload's shape (8 x 4096 tokens, H16, c=d=128, N8, top-2, shared) and
    one decode step on the decode workload's shape (256 sequences x H16,
    N16, top-2, shared, fp32 states resident), inputs drawn on the device with
    the delta recipe (unit keys, log_alpha = logsigmoid(N(0,1))/16 and
    beta = sigmoid(N(0,1)) per (token, head))."""
    import torch
    from sparse_state_linear_router_gb300 import binding
    stream = torch.cuda.current_stream(dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(3)

    def timed(fn, reps):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    res = {}
    w = synth.WORKLOADS["layer_bf16"]
    T = sum(w.lengths)
    x = delta_inputs(w, T, dev, gen=gen)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(w.lengths)]).astype(np.int32), device=dev)
    cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, w.top_k, 1, 1.0, "bf16")
    ws = torch.empty(binding.load().sse_delta_forward_workspace_size(binding.ctypes.byref(cfg), T, len(w.lengths)),
                     dtype=torch.uint8, device=dev)
    ms = timed(lambda: binding.delta_forward(cfg, x["q"], x["k"], x["v"], x["la"], x["b"], x["lg"], cu,
                                             workspace=ws), 3)
    res["forward_layer_shape"] = {"ms": ms, "tokens_per_s": T / (ms * 1e-3), "form": "chunked (tensor cores)",
                                  "workload": "8 x 4096 tokens, H16, c=d=128, N8, top-2, shared, bf16"}
    cfg_r = binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, w.top_k, 1, 1.0, "bf16",
                                "recurrent")
    ms = timed(lambda: binding.delta_forward(cfg_r, x["q"], x["k"], x["v"], x["la"], x["b"], x["lg"], cu,
                                             workspace=ws), 3)
    res["forward_layer_shape_token_serial"] = {"ms": ms, "tokens_per_s": T / (ms * 1e-3),
                                               "form": "token by token (CUDA cores)",
                                               "workload": "8 x 4096 tokens, H16, c=d=128, N8, top-2, shared, bf16"}
    del x, ws
    w = synth.WORKLOADS["decode_bf16"]
    B = w.decode_batch
    x = delta_inputs(w, B, dev, gen=gen)
    cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, w.top_k, 1, 1.0, "bf16")
    state = torch.zeros((B, w.num_heads, w.num_slots, w.key_dim, w.value_dim), dtype=torch.float32, device=dev)
    ms = timed(lambda: binding.delta_decode_step(cfg, state, x["q"], x["k"], x["v"], x["la"], x["b"], x["lg"]), 10)
    nbytes = decode_bytes(w, B)  # the same state traffic as the GLA decode: k + 1 states read and written
    res["decode_step"] = {"ms": ms, "tokens_per_s": B / (ms * 1e-3), "gbs": nbytes / (ms * 1e6),
                          "frac_of_hbm_peak": nbytes / (ms * 1e6) / _peaks()["hbm_gbs"],
                          "workload": "256 sequences x H16, c=d=128, N16, top-2, shared, fp32 states"}
    del x, state
    torch.cuda.empty_cache()
    return res


def run_native(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from sparse_state_linear_router_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        from sparse_state_linear_router_gb300 import build as libbuild
        libbuild.build()
    binding.load()
    do_fwd = args.part in ("both", "forward")
    do_dec = args.part in ("both", "decode")
    names = ("q", "k", "v", "g", "logits")
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    P_ = binding._ptr
    launches = {"n": 0}

    w_fwd, w_dec = synth.WORKLOADS[args.fwd_workload], synth.WORKLOADS[DEC_WORKLOAD]
    if args.decode_batch:  # a smaller decode batch (profiling captures)
        import dataclasses
        w_dec = dataclasses.replace(w_dec, decode_batch=args.decode_batch)
    fwd_inp = synth.make_forward_inputs(w_fwd, seed=rank)   # also the CPU-baseline sample
    T, S = fwd_inp.total_tokens, fwd_inp.num_seqs
    B = w_dec.decode_batch
    pool = min(args.warmup + args.steps, 64)
    dec_host = [synth.make_decode_inputs(w_dec, s) for s in range(pool if do_dec else 4)]

    if do_fwd:
        cfg_f = binding.make_config(w_fwd.num_heads, w_fwd.key_dim, w_fwd.value_dim, w_fwd.num_partitions,
                                    w_fwd.top_k, w_fwd.use_shared, 1.0, w_fwd.dtype, args.algo)
        f = {n: binding.to_device(getattr(fwd_inp, n), dev) for n in names}
        cu = torch.from_numpy(fwd_inp.cu_seqlens).to(dev)
        init = None if fwd_inp.init_state is None else torch.from_numpy(fwd_inp.init_state).to(dev)
        out = torch.empty((T, w_fwd.num_heads, w_fwd.value_dim), dtype=torch.bfloat16, device=dev)
        fin = torch.empty((S, w_fwd.num_heads, w_fwd.num_slots, w_fwd.key_dim, w_fwd.value_dim),
                          dtype=torch.float32, device=dev)
        wsp = binding.forward_workspace(cfg_f, T, S, dev)
    if do_dec:
        cfg_d = binding.make_config(w_dec.num_heads, w_dec.key_dim, w_dec.value_dim, w_dec.num_partitions,
                                    w_dec.top_k, w_dec.use_shared, 1.0, w_dec.dtype)
        dq = [{n: binding.to_device(getattr(x, n), dev) for n in names} for x in dec_host]
        state = torch.zeros((B, w_dec.num_heads, w_dec.num_slots, w_dec.key_dim, w_dec.value_dim),
                            dtype=torch.float32, device=dev)
        dout = torch.empty((B, w_dec.num_heads, w_dec.value_dim), dtype=torch.bfloat16, device=dev)

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)   # materialise the handles
        return evs

    def forward_call(src, stage_events=None, out_t=None):
        st, n = binding.sse_forward_timed(cfg_f, P_(src["q"]), P_(src["k"]), P_(src["v"]), P_(src["g"]),
                                          P_(src["logits"]), None, None, P_(cu), S, T, P_(init), P_(fin),
                                          P_(out if out_t is None else out_t), None, None, P_(wsp), wsp.numel(), sh,
                                          None if stage_events is None else [e.cuda_event for e in stage_events])
        binding._check(st, "sse_forward_timed")
        launches["n"] += n

    def decode_call(x, out_t=None):
        st = binding.sse_decode_step(cfg_d, P_(x["q"]), P_(x["k"]), P_(x["v"]), P_(x["g"]),
                                     P_(x["logits"]), None, None, B, P_(state),
                                     P_(dout if out_t is None else out_t), None, None, sh)
        binding._check(st, "sse_decode_step")
        launches["n"] += 1

    def barrier():
        rank_barrier(ws)

    def max_over_ranks(x):
        return max_over_ranks_of(x, ws, dev)

    # ---- device-resident timing -------------------------------------------
    for i in range(args.warmup):
        if do_fwd:
            forward_call(f)
        if do_dec:
            decode_call(dq[i % pool])
    torch.cuda.synchronize()
    fwd_ev = [new_events(4) for _ in range(args.steps)] if do_fwd else []
    dec_ev = [new_events(2) for _ in range(args.steps)] if do_dec else []
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    launches["n"] = 0
    with ClockSampler(local) as clk:
        time.sleep(0.15)
        # the timed steps: no event between the forward's kernels, so its
        # dependent launches overlap as they do in use
        t_start.record(stream)
        for i in range(args.steps):
            if do_fwd:
                forward_call(f)
            if do_dec:
                dec_ev[i][0].record(stream)
                decode_call(dq[(args.warmup + i) % pool])
                dec_ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        timed_launches = launches["n"]
        # the same forward calls again with an event at each stage boundary
        # (routing, main kernel + redo pass, combine): the per-stage breakdown
        for i in range(args.steps if do_fwd else 0):
            forward_call(f, fwd_ev[i])
        torch.cuda.synchronize()
        time.sleep(0.15)
    barrier()
    ms_step = max_over_ranks(t_start.elapsed_time(t_end)) / args.steps
    tokens_step = (T if do_fwd else 0) + (B if do_dec else 0)
    value = whole_job_tokens_per_s(ws, tokens_step, ms_step)

    peaks = _peaks()
    hbm = peaks["hbm_gbs"]
    has_init = fwd_inp.init_state is not None
    kernels, extra = {}, {}
    step_bytes = step_flops = 0
    if do_fwd:
        fwd_main_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in fwd_ev)
        fwd_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in fwd_ev)
        b_main = forward_main_bytes(w_fwd, T, S, init=has_init)
        kernels["forward_main"] = {"ms": fwd_main_ms, "bytes": b_main, "gbs": b_main / (fwd_main_ms * 1e6)}
        fb = forward_step_bytes(w_fwd, T, S, init=has_init)
        ff = forward_flops(w_fwd, T)
        step_bytes += fb
        step_flops += ff
        extra["forward"] = {
            "ms": fwd_ms, "route_ms": statistics.mean(e[0].elapsed_time(e[1]) for e in fwd_ev),
            "main_ms": fwd_main_ms, "tail_ms": statistics.mean(e[2].elapsed_time(e[3]) for e in fwd_ev),
            "tokens_per_s": T / (fwd_ms * 1e-3),
            "roofline_frac": max(ff / (peaks["bf16_tflops"] * 1e12), fb / (hbm * 1e9)) / (fwd_ms * 1e-3)}
    if do_dec:
        dec_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in dec_ev)
        b_dec = decode_bytes(w_dec, B)
        kernels["decode"] = {"ms": dec_ms, "bytes": b_dec, "gbs": b_dec / (dec_ms * 1e6)}
        step_bytes += b_dec
        step_flops += decode_flops(w_dec, B)
        extra["decode"] = {"ms": dec_ms, "tokens_per_s": B / (dec_ms * 1e-3),
                           "hbm_frac": (b_dec / (dec_ms * 1e-3)) / (hbm * 1e9)}
    dom_name = max(kernels, key=lambda kname: kernels[kname]["ms"])
    dom = kernels[dom_name]
    t_bind = max(step_flops / (peaks["bf16_tflops"] * 1e12), step_bytes / (hbm * 1e9))

    # ---- end to end through the C ABI with host buffers ---------------------
    # Every step copies its inputs from pinned host memory and its outputs back.
    # The copies run on their own streams into double-buffered device tensors,
    # so step i's inputs travel while step i-1 computes (a serving pipeline).
    e2e = None
    if not args.no_e2e:
        h2d = d2h = 0
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        ev_in, ev_done, ev_out = [ev(), ev()], [ev(), ev()], [ev(), ev()]
        if do_fwd:
            hf = {n: f[n].cpu().pin_memory() for n in names}
            dfs = [{n: torch.empty_like(f[n]) for n in names} for _ in range(2)]
            outs = [out, torch.empty_like(out)]
            hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
            h2d += sum(hf[n].numel() * hf[n].element_size() for n in names)
            d2h += hout.numel() * hout.element_size()
        if do_dec:
            hd = [{n: dq[i][n].cpu().pin_memory() for n in names} for i in range(min(pool, 8))]
            dds = [{n: torch.empty_like(dq[0][n]) for n in names} for _ in range(2)]
            douts = [dout, torch.empty_like(dout)]
            hdout = torch.empty(dout.shape, dtype=dout.dtype).pin_memory()
            h2d += sum(hd[0][n].numel() * hd[0][n].element_size() for n in names)
            d2h += hdout.numel() * hdout.element_size()

        def e2e_step(i):
            b = i % 2
            with torch.cuda.stream(s_in):  # inputs of step i (buffers last read by step i-2)
                if i >= 2:
                    s_in.wait_event(ev_done[b])
                if do_fwd:
                    for n in names:
                        dfs[b][n].copy_(hf[n], non_blocking=True)
                if do_dec:
                    x = hd[i % len(hd)]
                    for n in names:
                        dds[b][n].copy_(x[n], non_blocking=True)
                ev_in[b].record(s_in)
            stream.wait_event(ev_in[b])
            if i >= 2:
                stream.wait_event(ev_out[b])  # outputs of step i-2 copied out
            if do_fwd:
                forward_call(dfs[b], out_t=outs[b])
            if do_dec:
                decode_call(dds[b], out_t=douts[b])
            ev_done[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b])
                if do_fwd:
                    hout.copy_(outs[b], non_blocking=True)
                if do_dec:
                    hdout.copy_(douts[b], non_blocking=True)
                ev_out[b].record(s_out)

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(s_in)
        for i in range(args.steps):
            e2e_step(i)
        s_out.synchronize()
        eb.record(s_out)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(ea.elapsed_time(eb) / args.steps)
        e2e = {"value": whole_job_tokens_per_s(ws, tokens_step, e2e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "overlap": "inputs of step i copied on a second stream while step i-1 computes"}

    # ---- the other forward workloads (rank 0, N = 1, default run only) -------
    variants, variant_clocks, fig6, delta = None, None, None, None
    if do_fwd and do_dec and rank == 0 and ws == 1 and not args.no_variants:
        with ClockSampler(local) as vclk:
            variants = time_forward_variants(args, dev, peaks)
            fig6 = time_fwd_bwd_fig6(args, dev)
            delta = time_delta(args, dev)
        variant_clocks = vclk.summary()

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----------------------------
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        smp = OracleSampler(fwd_inp, w_fwd, dec_host[:4], w_dec, dec_seqs=16)
        t0 = time.perf_counter()
        smp.run_for(args.cpu_seconds)
        fwd_tps, dec_tps = smp.rates()
        if do_fwd and do_dec:
            cv = step_equivalent_tps(T, B, fwd_tps, dec_tps)
        else:
            cv = fwd_tps if do_fwd else dec_tps
        cpu = {"value": cv, "unit": "tokens/s", "cores": smp.threads, "kind": "oracle",
               "sample": smp.sample_text() + "; value = tokens/s of one full step at the measured rates",
               "seconds": round(time.perf_counter() - t0, 1)}

    if rank != 0:
        return 0
    # measured DRAM bytes of the dominant kernel (ncu, same workload and build)
    traffic, traffic_src = None, None
    if dom_name == "forward_main" and args.fwd_workload == FWD_WORKLOAD and args.algo in ("auto", "chunked"):
        traffic, summary = profiled_traffic("chunked_forward_kernel")
        if traffic is not None:
            traffic_src = f"ncu dram__bytes_read.sum + dram__bytes_write.sum, {summary}"
    parts = ([describe_forward(w_fwd, fwd_inp)] if do_fwd else []) + ([describe_decode(w_dec)] if do_dec else [])
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": " + ".join(parts),
            "fwd_tokens_per_step": T if do_fwd else 0, "decode_tokens_per_step": B if do_dec else 0,
            "algo": args.algo,
            "l2": "inputs larger than L2 (forward token tensors >= 545 MB, 4.6 GB decode states); no flush",
        },
        "roofline": {"kernel": dom_name, "bound": "hbm", "achieved": dom["gbs"], "peak": hbm,
                     "unit": "GB/s", "frac": dom["gbs"] / hbm, "traffic": traffic,
                     "traffic_source": traffic_src,
                     "peak_source": f"{peaks['source']} hbm_gbs (MEASURED_PEAKS.json)",
                     "algorithmic_bytes_per_launch": dom["bytes"], "avg_launch_ms": dom["ms"]},
        "kernels": {k_: {"avg_ms": v["ms"], "algorithmic_bytes": v["bytes"], "gbs": v["gbs"],
                         "frac_of_hbm_peak": v["gbs"] / hbm} for k_, v in kernels.items()},
        **extra,
        "step_roofline_frac": t_bind / (ms_step * 1e-3),
        "gpu_launches": timed_launches,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "e2e": e2e,
    }
    if variants is not None:
        line["forward_variants"] = variants
        line["fwd_bwd_fig6_shape"] = fig6
        line["delta_rule"] = delta
        line["forward_variants_clocks"] = variant_clocks
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def front_end_flops(w) -> int:
    """Tensor-core flops of one sse_front_end call: the projection GEMMs
    (q, k, v, g and the router logits) plus the shared LoRA's two factors."""
    T, D, H, c, d, N, r = w.tokens, w.hidden, w.num_heads, w.key_dim, w.value_dim, w.num_partitions, w.lora_rank
    main = 2 * T * D * H * (3 * c + d + N)
    lora = (2 * T * D * 2 * r + 2 * T * r * 2 * H * c) if r else 0
    return main + lora


def run_front_end(args):
    """One JSON line for the front end alone (sse_front_end on the
    32768-token, D = 2048 workload): tokens/s and its tensor-core roofline."""
    import torch
    from sparse_state_linear_router_gb300 import binding
    ws, rank, local = _dist()
    if ws > 1:
        raise SystemExit("--part front_end runs on one GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.FRONT_END_WORKLOADS["front_end_bf16"]
    inp = synth.make_front_end_inputs(w, seed=0)
    cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, 2, 1, 1.0, "bf16")
    dv = {n: (None if getattr(inp, n) is None else binding.to_device(getattr(inp, n), dev))
          for n in ("x", "w_q", "w_k", "w_v", "w_g", "w_e", "a_q", "b_q", "a_k", "b_k")}

    def call():
        return binding.front_end(cfg, dv["x"], dv["w_q"], dv["w_k"], dv["w_v"], dv["w_g"], dv["w_e"],
                                 a_q=dv["a_q"], b_q=dv["b_q"], a_k=dv["a_k"], b_k=dv["b_k"], outs=outs,
                                 workspace=wsp)
    outs, wsp = None, None
    first = call()
    outs = {n: first[n] for n in ("q", "k", "v", "log_gate", "logits", "q_shared", "k_shared")}
    wsp = first["workspace"]
    for _ in range(args.warmup):
        call()
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.15)
        ev[0].record(stream)
        for _ in range(args.steps):
            call()
        ev[1].record(stream)
        torch.cuda.synchronize()
        time.sleep(0.15)
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    st, flags = binding.sse_read_device_status(wsp.data_ptr(), binding._stream())
    peaks = _peaks()
    flops = front_end_flops(w)
    tflops = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]
    line = {
        "metric": "SSE front end tokens/s (projections, key softmax, log-gate, shared LoRA) on 1 GB300",
        "value": w.tokens / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name} (T={w.tokens}, D={w.hidden}, H{w.num_heads}, c={w.key_dim}, "
                               f"d={w.value_dim}, N{w.num_partitions}, LoRA rank {w.lora_rank})",
                   "l2": "weights (33 MB) stay in L2, x (134 MB) and outputs (0.81 GB) exceed it; no flush"},
        "roofline": {"kernel": "front_end_kernel", "bound": "tensor", "achieved": tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": tflops / peak, "traffic": None,
                     "peak_source": f"{peaks['source']} bf16_tflops (MEASURED_PEAKS.json)",
                     "algorithmic_flops_per_call": flops},
        "gpu_launches": 2 * args.steps,
        "device_flags": flags,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_delta(args):
    """One JSON line for sse_delta_forward alone (SSE on the gated delta rule,
    section 7d of the design notes) on the layer workload's shape, inputs as
    time_delta draws them: tokens/s of the forward and its time per call."""
    import torch
    from sparse_state_linear_router_gb300 import binding
    ws, rank, local = _dist()
    if ws > 1:
        raise SystemExit("--part delta runs on one GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS["layer_bf16"]
    T = sum(w.lengths)
    x = delta_inputs(w, T, dev, seed=3)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(w.lengths)]).astype(np.int32), device=dev)
    cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, w.num_partitions, w.top_k, 1, 1.0, "bf16")
    wsp = torch.empty(binding.load().sse_delta_forward_workspace_size(binding.ctypes.byref(cfg), T, len(w.lengths)),
                      dtype=torch.uint8, device=dev)

    def call():
        binding.delta_forward(cfg, x["q"], x["k"], x["v"], x["la"], x["b"], x["lg"], cu, workspace=wsp)
    for _ in range(args.warmup):
        call()
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.15)
        ev[0].record(stream)
        for _ in range(args.steps):
            call()
        ev[1].record(stream)
        torch.cuda.synchronize()
        time.sleep(0.15)
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    line = {
        "metric": "SSE on the gated delta rule: forward tokens/s on 1 GB300",
        "value": T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": "delta-rule forward, 8 x 4096 tokens, H16, c=d=128, N8, top-2, shared, "
                               "bf16 in, fp32 state"},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def run_backward(args, N=4, L=8192):
    """One JSON line for sse_backward alone at the operator shape of the
    pages' Fig. 6 (8 heads, head dim 128, top-1 of N = 4, shared,
    cu_seqlens = [0, L/2, L], bf16; d_out ~ N(0, 1), no final-state gradient):
    tokens/s of the backward and its time per call."""
    import dataclasses

    import torch
    from sparse_state_linear_router_gb300 import binding
    ws, rank, local = _dist()
    if ws > 1:
        raise SystemExit("--part backward runs on one GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = dataclasses.replace(synth.WORKLOADS["layer_bf16"], name=f"fig6_N{N}", num_heads=8, num_partitions=N,
                            top_k=1, lengths=(L // 2, L // 2), sigma_router=1.0)
    x = synth.make_forward_inputs_device(w, seed=0, device=dev)
    T, S = x["total_tokens"], x["num_seqs"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    d_out = torch.randn((T, w.num_heads, w.value_dim), generator=gen, device=dev).to(torch.bfloat16)
    cfg = binding.make_config(w.num_heads, w.key_dim, w.value_dim, N, 1, 1, 1.0, "bf16", args.algo)
    bws = torch.empty(binding.sse_backward_workspace_size(cfg, T, S), dtype=torch.uint8, device=dev)

    def call():
        binding.backward(cfg, x["q"], x["k"], x["v"], x["g"], x["logits"], x["cu_seqlens"], d_out,
                         want_d_initial_state=False, workspace=bws)
    for _ in range(args.warmup):
        call()
    stream = torch.cuda.current_stream()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.15)
        ev[0].record(stream)
        for _ in range(args.steps):
            call()
        ev[1].record(stream)
        torch.cuda.synchronize()
        time.sleep(0.15)
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    line = {
        "metric": "SSE backward tokens/s at Fig. 6's operator shape on 1 GB300",
        "value": T / (ms * 1e-3), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"backward, H8, c=d=128, top-1 of N={N}, shared, cu_seqlens=[0, {L // 2}, {L}], "
                               "bf16 in, fp32 state and slots", "algo": args.algo},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--algo", choices=["auto", "chunked", "recurrent", "masked"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--decode-batch", type=int, default=0,
                    help="decode sequences per step (default: the workload's 256; smaller for ncu captures)")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the forward-only timings of the other workloads (varlen, small, skewed)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--part", choices=["both", "forward", "decode", "front_end", "backward", "delta"],
                    default="both",
                    help="time the whole step (default), one of its two calls, the front end alone, the "
                         "backward at Fig. 6's shape, or the delta-rule forward on the layer shape")
    ap.add_argument("--fwd-workload", choices=["layer_bf16", "varlen_bf16", "small_bf16"],
                    default=FWD_WORKLOAD, help="forward batch of the step")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.part == "front_end":
        return run_front_end(args)
    if args.part == "backward":
        return run_backward(args)
    if args.part == "delta":
        return run_delta(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())

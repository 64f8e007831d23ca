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
device -> host copies of its outputs inside the timed region), SM clocks
sampled during the timed region, and the fp64 CPU oracle timed on a bounded
sample of the same workload (cpu_baseline).

``--impl reference`` times the CPU oracle alone on bounded samples of the same
workload (the reference arm of this build: the pages publish no code).
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
                 "--format=csv,noheader,nounits", "-lms", "100"],
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


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return 0
    w_fwd, w_dec = synth.WORKLOADS[FWD_WORKLOAD], synth.WORKLOADS[DEC_WORKLOAD]
    fwd_inp = synth.make_forward_inputs(w_fwd, seed=0)
    dec_steps = [synth.make_decode_inputs(w_dec, s, batch=16) for s in range(4)]
    T = fwd_inp.total_tokens
    B = w_dec.decode_batch
    smp = OracleSampler(fwd_inp, w_fwd, dec_steps, w_dec, dec_seqs=16)
    for _ in range(args.warmup):
        smp.once()
    smp.reset()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.once()
    wall = time.perf_counter() - t0
    fwd_tps, dec_tps = smp.rates()
    value = step_equivalent_tps(T, B, fwd_tps, dec_tps)
    threads = smp.threads
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{FWD_WORKLOAD} forward (8x4096 tokens, H16, c=d=128, N8, k2, shared) + "
                               f"{DEC_WORKLOAD} step (256 seqs, H16, c=d=128, N16, k2, shared)",
                   "fwd_tokens_per_step": T, "decode_tokens_per_step": B},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": "per step: " + smp.sample_text() + "; value = tokens/s of one full step "
                                                                       "at the measured forward and decode rates"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


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

    w_fwd, w_dec = synth.WORKLOADS[FWD_WORKLOAD], synth.WORKLOADS[DEC_WORKLOAD]
    fwd_inp = synth.make_forward_inputs(w_fwd, seed=rank)
    T, S = fwd_inp.total_tokens, fwd_inp.num_seqs
    B = w_dec.decode_batch
    nsteps = args.warmup + args.steps
    pool = min(nsteps, 64)
    dec_host = [synth.make_decode_inputs(w_dec, s) for s in range(pool)]
    cfg_f = binding.make_config(w_fwd.num_heads, w_fwd.key_dim, w_fwd.value_dim, w_fwd.num_partitions,
                                w_fwd.top_k, w_fwd.use_shared, 1.0, w_fwd.dtype, args.algo)
    cfg_d = binding.make_config(w_dec.num_heads, w_dec.key_dim, w_dec.value_dim, w_dec.num_partitions,
                                w_dec.top_k, w_dec.use_shared, 1.0, w_dec.dtype)
    names = ("q", "k", "v", "g", "logits")
    f = {n: binding.to_device(getattr(fwd_inp, n), dev) for n in names}
    cu = torch.from_numpy(fwd_inp.cu_seqlens).to(dev)
    H, d = w_fwd.num_heads, w_fwd.value_dim
    P = w_fwd.num_slots
    out = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((S, H, P, w_fwd.key_dim, d), dtype=torch.float32, device=dev)
    wsp = binding.forward_workspace(cfg_f, T, S, dev)
    dq = [{n: binding.to_device(getattr(x, n), dev) for n in names} for x in dec_host]
    state = torch.zeros((B, w_dec.num_heads, w_dec.num_slots, w_dec.key_dim, w_dec.value_dim),
                        dtype=torch.float32, device=dev)
    dout = torch.empty((B, w_dec.num_heads, w_dec.value_dim), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    P_ = binding._ptr

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)   # materialise the handles
        return evs

    launches = {"n": 0}

    def forward_call(fin_t, out_t, stage_events=None):
        st, n = binding.sse_forward_timed(cfg_f, P_(f["q"]), P_(f["k"]), P_(f["v"]), P_(f["g"]),
                                          P_(f["logits"]), None, None, P_(cu), S, T, None, P_(fin_t),
                                          P_(out_t), None, None, P_(wsp), wsp.numel(), sh,
                                          None if stage_events is None else [e.cuda_event for e in stage_events])
        binding._check(st, "sse_forward_timed")
        launches["n"] += n

    def decode_call(i, inputs=None):
        x = dq[i % pool] if inputs is None else inputs
        st = binding.sse_decode_step(cfg_d, P_(x["q"]), P_(x["k"]), P_(x["v"]), P_(x["g"]),
                                     P_(x["logits"]), None, None, B, P_(state), P_(dout), None, None, sh)
        binding._check(st, "sse_decode_step")
        launches["n"] += 1

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---- device-resident timing -------------------------------------------
    for i in range(args.warmup):
        forward_call(fin, out)
        decode_call(i)
    torch.cuda.synchronize()
    fwd_ev = [new_events(4) for _ in range(args.steps)]
    dec_ev = [new_events(2) for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier()
    launches["n"] = 0
    with ClockSampler(local) as clk:
        time.sleep(0.15)
        t_start.record(stream)
        for i in range(args.steps):
            forward_call(fin, out, fwd_ev[i])
            dec_ev[i][0].record(stream)
            decode_call(args.warmup + i)
            dec_ev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        time.sleep(0.15)
    barrier()
    timed_launches = launches["n"]
    elapsed_ms = t_start.elapsed_time(t_end)
    if ws > 1:
        import torch.distributed as dist
        tt = torch.tensor([elapsed_ms], device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        elapsed_ms = float(tt.item())
    ms_step = elapsed_ms / args.steps
    fwd_main_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in fwd_ev)
    fwd_route_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in fwd_ev)
    fwd_tail_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in fwd_ev)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[3]) for e in fwd_ev)
    dec_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in dec_ev)
    tokens_step = T + B
    value = ws * tokens_step / (ms_step * 1e-3)

    peaks = _peaks()
    hbm = peaks["hbm_gbs"]
    b_main = forward_main_bytes(w_fwd, T, S)
    b_dec = decode_bytes(w_dec, B)
    kernels = {
        "forward_main": {"ms": fwd_main_ms, "bytes": b_main, "gbs": b_main / (fwd_main_ms * 1e6)},
        "decode": {"ms": dec_ms, "bytes": b_dec, "gbs": b_dec / (dec_ms * 1e6)},
    }
    dom_name = max(kernels, key=lambda kname: kernels[kname]["ms"])
    dom = kernels[dom_name]
    step_bytes = forward_step_bytes(w_fwd, T, S) + b_dec
    step_flops = forward_flops(w_fwd, T) + decode_flops(w_dec, B)
    t_bind = max(step_flops / (peaks["bf16_tflops"] * 1e12), step_bytes / (hbm * 1e9))

    # ---- end to end through the C ABI with host buffers ---------------------
    e2e = None
    if not args.no_e2e:
        hf = {n: f[n].cpu().pin_memory() for n in names}
        hd = [{n: dq[i][n].cpu().pin_memory() for n in names} for i in range(min(pool, 8))]
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hdout = torch.empty(dout.shape, dtype=dout.dtype).pin_memory()
        df = {n: torch.empty_like(f[n]) for n in names}
        dd = {n: torch.empty_like(dq[0][n]) for n in names}
        h2d = sum(hf[n].numel() * hf[n].element_size() for n in names) + \
            sum(hd[0][n].numel() * hd[0][n].element_size() for n in names)
        d2h = hout.numel() * hout.element_size() + hdout.numel() * hdout.element_size()

        def e2e_step(i):
            for n in names:
                df[n].copy_(hf[n], non_blocking=True)
            st, _ = binding.sse_forward_timed(cfg_f, P_(df["q"]), P_(df["k"]), P_(df["v"]), P_(df["g"]),
                                              P_(df["logits"]), None, None, P_(cu), S, T, None, P_(fin),
                                              P_(out), None, None, P_(wsp), wsp.numel(), sh, None)
            binding._check(st, "sse_forward_timed")
            x = hd[i % len(hd)]
            for n in names:
                dd[n].copy_(x[n], non_blocking=True)
            decode_call(0, dd)
            hout.copy_(out, non_blocking=True)
            hdout.copy_(dout, non_blocking=True)

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(args.steps):
            e2e_step(i)
        b.record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = a.elapsed_time(b) / args.steps
        if ws > 1:
            import torch.distributed as dist
            tt = torch.tensor([e2e_ms], device=dev)
            dist.all_reduce(tt, op=dist.ReduceOp.MAX)
            e2e_ms = float(tt.item())
        e2e = {"value": ws * tokens_step / (e2e_ms * 1e-3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----------------------------
    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        smp = OracleSampler(fwd_inp, w_fwd, dec_host[:4], w_dec, dec_seqs=16)
        t0 = time.perf_counter()
        smp.run_for(args.cpu_seconds)
        fwd_tps, dec_tps = smp.rates()
        cpu = {"value": step_equivalent_tps(T, B, fwd_tps, dec_tps), "unit": "tokens/s",
               "cores": smp.threads, "kind": "oracle",
               "sample": smp.sample_text() + "; value = tokens/s of one full step at the measured rates",
               "seconds": round(time.perf_counter() - t0, 1)}

    if rank != 0:
        return 0
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {
            "workload": f"{FWD_WORKLOAD} forward (8 seqs x 4096 tokens, H16, c=d=128, N8, top-2, shared, "
                        f"bf16 in, fp32 state) + {DEC_WORKLOAD} step (256 seqs x H16, c=d=128, N16, top-2, "
                        f"shared, fp32 states resident)",
            "fwd_tokens_per_step": T, "decode_tokens_per_step": B, "algo": args.algo,
            "l2": "inputs larger than L2 (545 MB forward token tensors, 4.6 GB decode states); no flush",
        },
        "roofline": {"kernel": dom_name, "bound": "hbm", "achieved": dom["gbs"], "peak": hbm,
                     "unit": "GB/s", "frac": dom["gbs"] / hbm, "traffic": None,
                     "peak_source": f"{peaks['source']} hbm_gbs (MEASURED_PEAKS.json)",
                     "algorithmic_bytes_per_launch": dom["bytes"], "avg_launch_ms": dom["ms"]},
        "kernels": {k_: {"avg_ms": v["ms"], "algorithmic_bytes": v["bytes"], "gbs": v["gbs"],
                         "frac_of_hbm_peak": v["gbs"] / hbm} for k_, v in kernels.items()},
        "forward": {"ms": fwd_ms, "route_ms": fwd_route_ms, "main_ms": fwd_main_ms, "tail_ms": fwd_tail_ms,
                    "tokens_per_s": T / (fwd_ms * 1e-3),
                    "roofline_frac": max(forward_flops(w_fwd, T) / (peaks["bf16_tflops"] * 1e12),
                                         forward_step_bytes(w_fwd, T, S) / (hbm * 1e9)) / (fwd_ms * 1e-3)},
        "decode": {"ms": dec_ms, "tokens_per_s": B / (dec_ms * 1e-3),
                   "hbm_frac": (b_dec / (dec_ms * 1e-3)) / (hbm * 1e9)},
        "step_roofline_frac": t_bind / (ms_step * 1e-3),
        "gpu_launches": timed_launches,
        "clocks": clk.summary(),
        "cpu_baseline": cpu,
        "e2e": e2e,
    }
    print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--algo", choices=["auto", "chunked", "recurrent"], default="auto")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the KDA forward pass on GB300.

One step = one kda_fwd call over the fixed-length prefill workload
B=1, T=8192, H=96, K=V=128 (bf16 q/k/v/g/beta/out, bf16 initial state, fp32
final state; seeded synthetic inputs shaped like the FlashKDA H20 benchmark
on the pages).  Inputs are resident in HBM before the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun, one rank per GPU) every
rank runs its own replica of the workload (weak scaling: the (sequence, head)
recurrences are independent, so there is no collective on the data path);
time is the max over ranks.  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "prefill_t8192_h96"
METRIC = "KDA fwd tokens/s at T=8192 H=96 D=128 bf16; % of tensor/HBM roofline"
K = V = 128
C = 16
# Algorithmic work of the chunked method per (token, head):
#   flops: 6KV (state reads S^T q, S^T k-side w, state update) + 2C(3K + 2V)
#          (A_kk, A_qk, w; u and A_qk U)  = 118,784
#   bytes: q, k, g, v (2 B x 128 each), beta (2 B), out (2 B x 128) = 1,282
# plus, per (sequence, head), the initial state read and the final state write.
FLOP_PER_TH = 6 * K * V + 2 * C * (3 * K + 2 * V)
BYTES_PER_TH = 4 * 2 * 128 + 2 + 2 * 128
# Backward pass (kda_bwd), token-level reverse of the recurrence on CUDA cores, per
# (token, head): the forward step it recomputes (S' = Diag(a) S, r = S'^T k, S += k d^T:
# 5KV) and the reverse step (dS += q dO^T, dq, dd, dk, dS', dk += S' dr, da, dS = a dS':
# 15KV) -- 20KV flop; bytes: q, k, v, g, dO and beta read (bf16), dq, dk, dv, dg and
# dbeta written (fp32).  It is bound by fp32 CUDA-core arithmetic: the peak is 152 SMs
# x 128 fp32 lanes x 2 flop (a multiply-add) x 2.07 GHz.
BWD_FLOP_PER_TH = 20 * K * V
BWD_BYTES_PER_TH = 5 * 2 * 128 + 2 + 4 * 4 * 128 + 4
ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
BWD_WORKLOAD = "bwd_prefill_t8192_h96"
# The fused kernel does the whole path, so its algorithmic work is the path's.
KERNEL_FLOP_PER_TH = {"fused_kernel": FLOP_PER_TH}
KERNEL_BYTES_PER_TH = {"fused_kernel": BYTES_PER_TH}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "of measured"
    return 6800.0, 1900.0, "of fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        # raw samples go to KDA_BENCH_CLOCKS_DIR (default: the system temp directory);
        # the JSON line carries their summary
        out_dir = os.environ.get("KDA_BENCH_CLOCKS_DIR", tempfile.gettempdir())
        self.path = os.path.join(out_dir, f"clocks_gpu{gpu_index}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for ln in open(self.path):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "N/A") else 0.0,
                             "hw": parts[5], "hwt": parts[6], "swt": parts[7], "pcap": parts[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        mx = max(r["max"] for r in rows)
        loaded = [r for r in rows if r["power"] > 0.2 * max(x["power"] for x in rows)] or rows
        reasons = []
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                          ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
            if any(r[key].lower() == "active" for r in loaded):
                reasons.append(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded), "sm_max_mhz": mx,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl != "reference" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def max_over_ranks(pg, x: float, device=None) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device if device is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def source_digest(*names) -> str:
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "gated_delta_rule_39_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str | None = None):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if the kernel's
    source has not changed since the capture and (when given) the capture was taken on
    `workload`; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    if rec.get("source_digest") != source_digest(*rec.get("sources", [])):
        return None
    if workload is not None and rec.get("workload_name") != workload:
        return None
    return rec.get("bytes_per_launch")


# ---------------------------------------------------------------------------
# The other workloads of the pages' benchmark reported in the same line (each a
# nested object with its own timing, roofline and CPU-oracle sample).
OTHER_WORKLOADS = ("prefill_t8192_h64", "varlen_mixed_t8192_h96", "varlen_uniform_8x1024_h96",
                   "carry_t65536_h32", "varlen_short_20000_h16")


def algorithmic_work(d, calls):
    """(bytes, flops, token-heads) of one step: every kda_fwd call of the step moves its
    inputs and outputs once, plus each call's state read (if any) and write."""
    B, T, H, _ = d["q"].shape
    N = d["N"]
    th = B * T * H
    s0 = d.get("initial_state")
    init_b = 0 if s0 is None else (2 if s0.dtype == np.uint16 else 4)
    w = d.get("workload")
    fd = "f32" if w is None else w.final_dtype
    write_b = 0 if fd is None else (4 if fd == "f32" else 2)
    state_bytes = 0
    for i in range(calls):
        read_b = init_b if i == 0 else 4      # later calls read the carried fp32 state
        last = i == calls - 1
        state_bytes += N * H * K * V * (read_b + (write_b if last else 4))
    return BYTES_PER_TH * th + state_bytes, FLOP_PER_TH * th, th


def roofline_of(kernel, ms, bytes_, flop, hbm, tflops, src, alu=False):
    t_hbm = bytes_ / (hbm * 1e9)
    t_tc = flop / (tflops * 1e12)
    if alu and flop / (ALU_TFLOPS * 1e12) >= t_hbm:
        roof = {"bound": "alu", "achieved": flop / (ms * 1e-3) / 1e12, "peak": ALU_TFLOPS,
                "unit": "TFLOP/s", "frac": flop / (ms * 1e-3) / 1e12 / ALU_TFLOPS,
                "kernel": kernel, "kernel_ms": ms,
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flop x 2.07 GHz"}
        return roof
    if t_tc >= t_hbm:
        roof = {"bound": "tensor", "achieved": flop / (ms * 1e-3) / 1e12, "peak": tflops,
                "unit": "TFLOP/s"}
    else:
        roof = {"bound": "hbm", "achieved": bytes_ / (ms * 1e-3) / 1e9, "peak": hbm, "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["kernel"] = kernel
    roof["kernel_ms"] = ms
    roof["peak_source"] = src
    return roof


class Runner:
    """Device copies of one workload and the call sequence of one step."""

    def __init__(self, d, device, stream, segments=0):
        import torch
        import gated_delta_rule_39_gb300 as kda
        self.kda = kda
        self.d = d
        self.stream = stream
        self.segments = segments   # 0: kda_fwd's own choice; else kda_fwd_segments
        B, T, H, _ = d["q"].shape
        self.B, self.T, self.H, self.N = B, T, H, d["N"]

        def bf16(bits):
            return (torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
                    .view(torch.bfloat16))

        self.x = {n: bf16(d[n]) for n in ("q", "k", "v", "g", "beta")}
        self.A_log = torch.from_numpy(d["A_log"]).to(device)
        self.dt_bias = torch.from_numpy(d["dt_bias"]).to(device)
        s0 = d.get("initial_state")
        self.s0 = None if s0 is None else (bf16(s0) if s0.dtype == np.uint16
                                           else torch.from_numpy(s0).to(device))
        cu = d.get("cu_seqlens")
        self.cu = None if cu is None else torch.from_numpy(cu.astype(np.int32)).to(device)
        self.out = torch.empty((B, T, H, V), dtype=torch.bfloat16, device=device)
        w = d.get("workload")
        fd = "f32" if w is None else w.final_dtype   # None: the call writes no final state
        self.s1 = (None if fd is None else
                   torch.empty((self.N, H, K, V), device=device,
                               dtype=torch.float32 if fd == "f32" else torch.bfloat16))
        self.calls = w.carry_calls if w is not None else 1
        if self.calls > 1:   # one sequence cut into `calls` pieces, the state carried
            L = T // self.calls
            sl = lambda t, a: t[:, a * L:(a + 1) * L]
            self.pieces = [{n: sl(self.x[n], i) for n in self.x} for i in range(self.calls)]
            self.opieces = [sl(self.out, i) for i in range(self.calls)]
            self.carry = torch.empty_like(self.s1)

    def step(self):
        kda, x, d = self.kda, self.x, self.d
        seg = {} if self.segments == 0 or self.cu is not None else {"num_segments": self.segments}
        fwd = kda.kda_fwd_segments if seg else kda.kda_fwd
        if self.calls == 1:
            fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], self.out,
                self.A_log, self.dt_bias, d["lower_bound"], initial_state=self.s0,
                final_state=self.s1, cu_seqlens=self.cu, stream=self.stream, **seg)
            return
        for i, xp in enumerate(self.pieces):
            fwd(xp["q"], xp["k"], xp["v"], xp["g"], xp["beta"], d["scale"],
                self.opieces[i], self.A_log, self.dt_bias, d["lower_bound"],
                initial_state=(self.s0 if i == 0 else self.carry),
                final_state=(self.s1 if i == self.calls - 1 else self.carry),
                stream=self.stream, **seg)


class DecodeRunner:
    """One kda_decode step over N sequences x H heads, fp32 states updated in place."""

    def __init__(self, d, device, stream):
        import torch
        import gated_delta_rule_39_gb300 as kda
        self.kda = kda
        self.d = d
        self.stream = stream
        N, T, H, _ = d["q"].shape
        assert T == 1
        self.B, self.T, self.H, self.N = N, 1, H, N
        self.calls = 1

        def bf16(bits, shape):
            return (torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
                    .view(torch.bfloat16).reshape(shape))

        self.x = {n: bf16(d[n], (N, H, 128)) for n in ("q", "k", "v", "g")}
        self.x["beta"] = bf16(d["beta"], (N, H))
        self.A_log = torch.from_numpy(d["A_log"]).to(device)
        self.dt_bias = torch.from_numpy(d["dt_bias"]).to(device)
        self.state = torch.from_numpy(d["initial_state"]).to(device)
        self.out = torch.empty((N, H, V), dtype=torch.bfloat16, device=device)

    def step(self):
        x, d = self.x, self.d
        self.kda.kda_decode(x["q"], x["k"], x["v"], x["g"], x["beta"], d["scale"], self.out,
                            self.A_log, self.dt_bias, d["lower_bound"], state_in=self.state,
                            state_out=self.state, stream=self.stream)


DECODE_WORKLOAD = "decode_n256_h96"


class BwdRunner:
    """One kda_bwd call on the headline workload's inputs, a seeded dL/d(out) and
    dL/d(final state); outputs allocated once."""

    def __init__(self, d, device, stream, seed):
        import ctypes
        import torch
        import synth
        import gated_delta_rule_39_gb300 as kda
        self.kda = kda
        self.lib = kda.load_library()
        self.d = d
        self.stream = stream
        B, T, H, _ = d["q"].shape
        self.B, self.T, self.H, self.N = B, T, H, d["N"]
        self.calls = 1

        def bf16(bits):
            return (torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device)
                    .view(torch.bfloat16))

        rng = np.random.default_rng(seed + 1000)
        self.x = {n: bf16(d[n]) for n in ("q", "k", "v", "g", "beta")}
        self.x["dout"] = bf16(synth.f32_to_bf16_bits(rng.standard_normal(d["v"].shape,
                                                                          dtype=np.float32)))
        self.dfinal = torch.from_numpy(rng.standard_normal((self.N, H, K, V), dtype=np.float32)).to(device)
        self.A_log = torch.from_numpy(d["A_log"]).to(device)
        self.dt_bias = torch.from_numpy(d["dt_bias"]).to(device)
        s0 = d.get("initial_state")
        self.s0 = None if s0 is None else (bf16(s0) if s0.dtype == np.uint16
                                           else torch.from_numpy(s0).to(device))
        f32 = dict(dtype=torch.float32, device=device)
        self.o = [torch.empty((B, T, H, K), **f32), torch.empty((B, T, H, K), **f32),
                  torch.empty((B, T, H, V), **f32), torch.empty((B, T, H, K), **f32),
                  torch.empty((B, T, H), **f32), torch.empty((H,), **f32),
                  torch.empty((H, K), **f32), torch.empty((self.N, H, K, V), **f32)]
        p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
        self.args = ([p(self.x[n]) for n in ("q", "k", "v", "g", "beta")] +
                     [ctypes.c_float(d["scale"]), p(self.A_log), p(self.dt_bias),
                      ctypes.c_float(d["lower_bound"]), p(self.s0),
                      0 if s0 is None or s0.dtype == np.uint16 else 1, p(self.x["dout"]),
                      p(self.dfinal)] + [p(t) for t in self.o] +
                     [None, 0, B, T, H, K, V, ctypes.c_void_p(stream.cuda_stream)])

    def step(self):
        rc = self.lib.kda_bwd(*self.args)
        if rc != 0:
            raise RuntimeError(f"kda_bwd failed: {self.kda.kda_status_string(rc)}")


def make_decode_inputs(seed):
    import synth
    return synth.make_inputs(256, 1, 96, seed=seed, init_dtype="f32")


def timed_steps(runner, steps, warmup, pg=None, device=None, sampler=None):
    """Warm up, then time `steps` steps with CUDA events on the launch stream; returns
    (elapsed ms, {kernel: (total ms, launches)})."""
    import torch
    kda = runner.kda
    for _ in range(warmup):
        runner.step()
    torch.cuda.synchronize(device)
    err = kda.kda_fwd_get_error(runner.stream)
    if err != 0:
        raise RuntimeError(f"device error after warm-up: {kda.kda_status_string(err)}")
    if sampler:
        sampler.__enter__()
    kda.kda_profile_enable(True)
    barrier(pg, device)
    torch.cuda.synchronize(device)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(runner.stream)
    for _ in range(steps):
        runner.step()
    ev1.record(runner.stream)
    torch.cuda.synchronize(device)
    barrier(pg, device)
    elapsed_ms = ev0.elapsed_time(ev1)
    prof = kda.kda_profile_read()
    kda.kda_profile_enable(False)
    if sampler:
        sampler.__exit__(None, None, None)
    return elapsed_ms, prof


def workload_line(name, d, elapsed_ms, prof, steps, world, calls, decode=False, bwd=False):
    """Throughput and roofline of one workload from its timing."""
    hbm, tflops, src = peaks()
    B, T, H, _ = d["q"].shape
    bytes_, flop, th = algorithmic_work(d, calls)
    if decode:   # the state is read and written in fp32 once per (sequence, head)
        bytes_ = B * H * (BYTES_PER_TH + K * V * (4 + 4))
        flop = B * H * 8 * K * V   # decay, S'^T k, update, S^T q: 4 multiply-adds per element
    if bwd:      # initial state read, dL/d(final state) read, d(initial state) written
        s0 = d.get("initial_state")
        init_b = 0 if s0 is None else (2 if s0.dtype == np.uint16 else 4)
        bytes_ = th * BWD_BYTES_PER_TH + d["N"] * H * K * V * (init_b + 4 + 4)
        flop = th * BWD_FLOP_PER_TH
    tokens_per_step = B * T
    dom = max(prof, key=lambda n: prof[n][0])
    # the dominant kernel's device time per step (a split call launches it twice)
    dom_ms = prof[dom][0] / steps
    ms_per_step = elapsed_ms / steps
    roof = (roofline_of(dom, dom_ms, bytes_, flop, hbm, tflops, src, alu=bwd)
            if dom in ("fused_kernel", "decode_kernel", "bwd_kernel") else None)
    if roof is not None:
        roof["traffic"] = ncu_traffic(dom, name)
    t_roof = max(bytes_ / (hbm * 1e9), flop / (tflops * 1e12))
    return {
        "workload": name, "value": world * tokens_per_step * steps / (elapsed_ms / 1e3),
        "unit": "tokens/s", "ms_per_step": ms_per_step, "calls_per_step": calls,
        "roofline": roof,
        "path_roofline": {"bound": "hbm" if bytes_ / (hbm * 1e9) >= flop / (tflops * 1e12) else "tensor",
                          "roofline_ms": t_roof * 1e3, "measured_ms": ms_per_step,
                          "frac": t_roof * 1e3 / ms_per_step, "bytes": bytes_, "flop": flop,
                          "peak_source": src},
        "kernel_ms": {n: (ms / max(1, c)) for n, (ms, c) in prof.items() if c},
        "gpu_launches": sum(c for _, c in prof.values()),
    }


def run_cuda(args, world, rank, local, pg):
    import torch

    import synth
    import gated_delta_rule_39_gb300 as kda

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    kda.load_library()
    stream = torch.cuda.current_stream(device)
    name = args.workload
    decode = name == DECODE_WORKLOAD
    if decode:
        d = make_decode_inputs(rank)
        runner = DecodeRunner(d, device, stream)
    else:
        if args.heads or args.tokens:
            w = synth.WORKLOADS[name]
            d = synth.make_inputs(w.B, args.tokens or w.T, args.heads or w.H, seed=rank,
                                  init_dtype=w.init_dtype)
        else:
            d = synth.make_workload(name, seed=rank)
        runner = (BwdRunner(d, device, stream, rank) if args.bwd
                  else Runner(d, device, stream, args.segments))
    B, T, H, N = runner.B, runner.T, runner.H, runner.N

    # ---- timed region: K steps, launch timing on the launch stream -------------
    sampler = ClockSampler(local) if rank == 0 else None
    elapsed_ms, prof = timed_steps(runner, args.steps, args.warmup, pg, device, sampler)
    elapsed_ms = max_over_ranks(pg, elapsed_ms, device)
    # a profiling case (another size, or the backward) has no traffic record of its own
    profiling = bool(args.heads or args.tokens or args.bwd)
    main = workload_line(name + " (profiling)" if profiling else name, d, elapsed_ms, prof,
                         args.steps, world, runner.calls, decode, bwd=args.bwd)

    # ---- end-to-end through the host-buffer entry point ---------------------------
    e2e = None
    if not args.no_e2e and runner.calls == 1 and not decode and not args.bwd:
        hx = {n: torch.from_numpy(np.ascontiguousarray(d[n]).view(np.int16)).view(torch.bfloat16)
              .pin_memory() for n in ("q", "k", "v", "g", "beta")}
        s0 = d.get("initial_state")
        hs0 = None if s0 is None else (
            torch.from_numpy(np.ascontiguousarray(s0).view(np.int16)).view(torch.bfloat16).pin_memory()
            if s0.dtype == np.uint16 else torch.from_numpy(s0).pin_memory())
        hA = torch.from_numpy(d["A_log"]).pin_memory()
        hdt = torch.from_numpy(d["dt_bias"]).pin_memory()
        hcu = None if d.get("cu_seqlens") is None else torch.from_numpy(
            d["cu_seqlens"].astype(np.int32))
        hout = torch.empty((B, T, H, V), dtype=torch.bfloat16).pin_memory()
        hs1 = torch.empty((N, H, K, V), dtype=torch.float32).pin_memory()

        def host_step():
            kda.kda_fwd_host(hx["q"], hx["k"], hx["v"], hx["g"], hx["beta"], d["scale"], hout,
                             hA, hdt, d["lower_bound"], initial_state=hs0, final_state=hs1,
                             cu_seqlens=hcu, stream=stream, device=device)

        host_step()
        e2e_steps = max(1, min(args.steps, 5))
        barrier(pg, device)
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            host_step()
        t1 = time.perf_counter()
        e2e_s = max_over_ranks(pg, t1 - t0, device)
        h2d = sum(t.numel() * t.element_size() for t in hx.values()) + hA.numel() * 4 + hdt.numel() * 4
        if hs0 is not None:
            h2d += hs0.numel() * hs0.element_size()
        if hcu is not None:
            h2d += hcu.numel() * 4
        d2h = hout.numel() * 2 + hs1.numel() * 4
        e2e = {"value": world * B * T * e2e_steps / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "entry_point": "kda_fwd_host"}

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only) -----------------------
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = (cpu_baseline_bwd(runner, target_s=args.cpu_seconds) if args.bwd
               else cpu_baseline(d, name, target_s=args.cpu_seconds))

    clocks = sampler.summary() if sampler else None

    # ---- the pages' other workloads, one nested object each (rank 0 prints) --------
    others = {}
    if (not args.heads and not args.tokens and not args.bwd and not args.no_other_workloads
            and name == WORKLOAD):
        for other in OTHER_WORKLOADS:
            od = synth.make_workload(other, seed=rank)
            orun = Runner(od, device, stream)
            ems, oprof = timed_steps(orun, max(3, args.steps // 2), 3, pg, device)
            ems = max_over_ranks(pg, ems, device)
            rec = workload_line(other, od, ems, oprof, max(3, args.steps // 2), world, orun.calls)
            rec["steps"] = max(3, args.steps // 2)
            rec["warmup"] = 3
            if world == 1 and not args.no_cpu_baseline:
                rec["cpu_baseline"] = cpu_baseline(od, other, target_s=args.cpu_seconds / 4)
            others[other] = rec
            del orun
            torch.cuda.empty_cache()
        # one decode step over a serving-sized batch (states in HBM, updated in place)
        dd = make_decode_inputs(rank)
        drun = DecodeRunner(dd, device, stream)
        ems, dprof = timed_steps(drun, args.steps, 3, pg, device)
        ems = max_over_ranks(pg, ems, device)
        rec = workload_line(DECODE_WORKLOAD, dd, ems, dprof, args.steps, world, 1, decode=True)
        rec["steps"], rec["warmup"] = args.steps, 3
        rec["config"] = {"N": 256, "H": 96, "K": K, "V": V, "state": "f32 in place",
                         "entry_point": "kda_decode"}
        if world == 1 and not args.no_cpu_baseline:
            rec["cpu_baseline"] = cpu_baseline(dd, DECODE_WORKLOAD, target_s=args.cpu_seconds / 8)
        others[DECODE_WORKLOAD] = rec
        del drun
        torch.cuda.empty_cache()
        # the backward pass over the headline workload (dL/d(out) and dL/d(final state)
        # drawn with the rank's seed)
        brun = BwdRunner(d, device, stream, rank)
        bsteps = max(3, args.steps // 4)
        ems, bprof = timed_steps(brun, bsteps, 3, pg, device)
        ems = max_over_ranks(pg, ems, device)
        rec = workload_line(BWD_WORKLOAD, d, ems, bprof, bsteps, world, 1, bwd=True)
        rec["steps"], rec["warmup"] = bsteps, 3
        rec["config"] = {"inputs": WORKLOAD, "d_out": "bf16 N(0,1)", "d_final_state": "f32 N(0,1)",
                         "entry_point": "kda_bwd", "outputs": "fp32 gradients"}
        if world == 1 and not args.no_cpu_baseline:
            rec["cpu_baseline"] = cpu_baseline_bwd(brun, target_s=args.cpu_seconds / 4)
        others[BWD_WORKLOAD] = rec
        del brun
        torch.cuda.empty_cache()

    if rank == 0:
        if args.heads or args.tokens or args.bwd:
            line_workload = (f"{'backward of ' if args.bwd else ''}{name} with T={T}, H={H} "
                             "(profiling case, not a bench line)")
        else:
            line_workload = name
        s0 = d.get("initial_state")
        line = {"metric": METRIC, "value": main["value"], "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": main["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "compute": "f16 and tf32 tensor-core MMA, f32 accumulate",
                "data": "synthetic (seeded; shapes of the pages' T=8192 H=96 D=128 benchmark)",
                "config": {"workload": line_workload, "B": B, "T": T, "H": H, "K": K, "V": V,
                           "initial_state": (None if s0 is None else
                                             ("bf16" if s0.dtype == np.uint16 else "f32")),
                           "final_state": "f32",
                           "l2": "inputs larger than L2 (1.02 GB read+written per step vs "
                                 "126 MB L2); no flush",
                           "parallelism": f"replicas x{world}"},
                "roofline": main["roofline"], "path_roofline": main["path_roofline"],
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": main["gpu_launches"],
                "kernel_ms": main["kernel_ms"], "clocks": clocks}
        if args.segments:
            line["config"]["segments"] = args.segments
        if others:
            line["workloads"] = others
        print(json.dumps(line), flush=True)


def cpu_baseline(d, workload: str = WORKLOAD, target_s: float = 12.0):
    """Time the fp64 oracle on a subset of heads (all tokens) of the same inputs."""
    import oracle
    H = d["q"].shape[2]
    T = d["q"].shape[1]
    threads = oracle.default_threads()
    # the oracle works on float64 copies; convert once outside the timing
    conv = {n: oracle.bf16_bits_to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")}
    s0 = d.get("initial_state")
    if s0 is not None:
        s0 = oracle.bf16_bits_to_f64(s0) if s0.dtype == np.uint16 else s0.astype(np.float64)

    def run(heads):
        t0 = time.perf_counter()
        oracle.kda_fwd(conv["q"], conv["k"], conv["v"], conv["g"], conv["beta"], d["scale"],
                       d["A_log"], d["dt_bias"], d["lower_bound"], initial_state=s0,
                       cu_seqlens=d.get("cu_seqlens"), heads=heads, n_threads=threads)
        return time.perf_counter() - t0

    probe = min(H, threads)
    t_probe = run(list(range(probe)))
    n_heads = int(min(H, max(probe, round(probe * target_s / max(t_probe, 1e-3)))))
    if n_heads > probe:
        t = run(list(range(n_heads)))
    else:
        n_heads, t = probe, t_probe
    tokens_equiv = d["q"].shape[0] * T * n_heads / H
    rec = {"value": tokens_equiv / t, "unit": "tokens/s", "cores": min(threads, n_heads),
           "kind": "oracle",
           "sample": f"{n_heads} of {H} heads x {d['q'].shape[0] * T} tokens of {workload}; "
                     f"tokens/s counts "
                     f"a token as all {H} heads ({t:.1f} s)"}
    if d.get("cu_seqlens") is None and d["q"].shape[0] == 1 and T >= 1024:
        # one thread on the first 1,024 tokens of head 0, extrapolated to all heads
        sl = {n: conv[n][:, :1024] for n in conv}
        t0 = time.perf_counter()
        oracle.kda_fwd(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], d["scale"], d["A_log"],
                       d["dt_bias"], d["lower_bound"], initial_state=s0, heads=[0], n_threads=1)
        t1 = time.perf_counter() - t0
        rec["one_thread"] = {"value": 1024 / H / t1, "unit": "tokens/s", "cores": 1,
                             "sample": f"first 1024 tokens of head 0 ({t1:.2f} s), "
                                       f"extrapolated: a token counts as all {H} heads"}
    return rec


def cpu_baseline_bwd(brun, target_s: float = 3.0):
    """Time the fp64 backward oracle on a subset of heads of the backward's inputs."""
    import oracle
    d = brun.d
    H = d["q"].shape[2]
    T = d["q"].shape[1]
    threads = oracle.default_threads()
    dout = brun.x["dout"].view(torch_int16()).cpu().numpy().view(np.uint16)
    dfinal = brun.dfinal.cpu().numpy()

    def run(heads):
        t0 = time.perf_counter()
        oracle.kda_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["scale"], d["A_log"],
                       d["dt_bias"], d["lower_bound"], dout, initial_state=d.get("initial_state"),
                       dfinal=dfinal, cu_seqlens=d.get("cu_seqlens"), heads=heads,
                       n_threads=threads)
        return time.perf_counter() - t0

    probe = min(H, threads)
    t_probe = run(list(range(probe)))
    n_heads = int(min(H, max(probe, round(probe * target_s / max(t_probe, 1e-3)))))
    if n_heads > probe:
        t = run(list(range(n_heads)))
    else:
        n_heads, t = probe, t_probe
    tokens_equiv = d["q"].shape[0] * T * n_heads / H
    return {"value": tokens_equiv / t, "unit": "tokens/s", "cores": min(threads, n_heads),
            "kind": "oracle",
            "sample": f"backward of {n_heads} of {H} heads x {d['q'].shape[0] * T} tokens; "
                      f"tokens/s counts a token as all {H} heads ({t:.1f} s)"}


def torch_int16():
    import torch
    return torch.int16


def run_reference(args, world, rank, local, pg):
    """The base contract's reference arm: here the fp64 CPU oracle, on rank 0."""
    if rank != 0:
        return
    import synth
    import oracle
    d = synth.make_workload(WORKLOAD, seed=0)
    H = d["q"].shape[2]
    T = d["q"].shape[1]
    threads = oracle.default_threads()
    conv = {n: oracle.bf16_bits_to_f64(d[n]) for n in ("q", "k", "v", "g", "beta")}
    s0 = oracle.bf16_bits_to_f64(d["initial_state"])
    heads_per_step = min(H, threads)

    def step():
        oracle.kda_fwd(conv["q"], conv["k"], conv["v"], conv["g"], conv["beta"], d["scale"],
                       d["A_log"], d["dt_bias"], d["lower_bound"], initial_state=s0,
                       heads=list(range(heads_per_step)), n_threads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    t = time.perf_counter() - t0
    value = T * heads_per_step / H * args.steps / t
    sample = (f"{heads_per_step} of {H} heads x {T} tokens of {WORKLOAD} per step; tokens/s "
              f"counts a token as all {H} heads")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": 1, "T": T, "H": H, "K": K, "V": V,
                   "initial_state": "bf16", "final_state": "f32",
                   "l2": "inputs larger than L2 (1.02 GB read+written per step vs 126 MB L2); "
                         "no flush",
                   "parallelism": f"replicas x{world}"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--heads", type=int, default=0,
                    help="profiling only: run the workload with this many heads instead")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling only: run the workload with this many tokens instead")
    ap.add_argument("--bwd", action="store_true",
                    help="profiling only: time the backward pass (kda_bwd) on the workload's "
                         "inputs instead of the forward")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="time this workload instead of the headline one (profiling)")
    ap.add_argument("--segments", type=int, default=0,
                    help="sequence split of fixed-length calls: 0 = kda_fwd's own choice, "
                         "1 = one pass, s = s segments (kda_fwd_segments)")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the nested measurements of the other workloads")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "cuda":
        print("note: warm-up raised to 3 steps", file=sys.stderr)
        args.warmup = 3
    world, rank, local, pg = dist_setup(args)
    if args.gpus != world and world > 1:
        print(f"note: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank, local, pg)
        else:
            run_cuda(args, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    main()

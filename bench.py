"""Benchmark of the B300 attention hot path (prints ONE JSON line on rank 0).

Headline workload: 14B-shaped 720p self-attention forward with 3D RoPE,
B = 1, grid 21x45x80 = 75,600 tokens, H = 40, d = 128, bf16 N(0,1) inputs.
A step is one wan_attn_fwd call (K RoPE pre-pass + attention kernel) on
inputs already resident in HBM; the RoPE tables are a per-grid constant built
once before timing. value = 4*B*H*L^2*d / step time (TFLOP/s).

Also reported (same run, under "also"): the tiny forward's latency, the
480p 1.3B self-attention forward, the cross-attention forward, the 64^3
training step (forward + backward), the VAE Conv3d and time-downsampling
layers, the FP8 forward, the decoupled text + image cross-attention and the
720p forward as two Ring steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own independent copy of the workload
(weak scaling; the path has no data exchange between ranks), and the step
time is the max over ranks. `--impl reference` times the fp64 CPU oracle on
a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)

METRIC = "attention TFLOP/s (bf16 fwd/bwd) at 32,760 and 75,600 tokens; % of dense BF16 peak"
# Lines for the VAE layer (--workload wan_vae_conv3d_*), a secondary workload.
CONV_METRIC = "causal Conv3d TFLOP/s (bf16, 2 FLOP per multiply-add); % of dense BF16 peak"
CONV_KINDS = ("conv3d", "time_down")
L2_BYTES = 126 * 2 ** 20


def _peaks():
    try:
        with open(os.path.join(HERE, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p["bf16_tflops_sustained"], "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ---------------------------------------------------------------------------
# Clock sampling during the timed region


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        return self.summary(self.lines)

    @staticmethod
    def merge(samplers):
        """Clock summary over the samples of several timed regions."""
        if all(s.proc is None for s in samplers):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        return ClockSampler.summary([ln for s in samplers for ln in s.lines])

    @staticmethod
    def summary(lines):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Distributed plumbing (timing only: barrier and max over ranks)


def dist_setup(n_gpus: int, gpu: bool = True):
    """Process group for N > 1 ranks: NCCL for the GPU arm, gloo for the
    reference arm (which runs on the host cores and needs no GPU)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = os.environ.get("WAN_BENCH_BACKEND", "nccl" if gpu else "gloo")
        if backend == "nccl":
            import torch

            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: units all ranks processed / slowest rank's time."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# Our arm


def timing_pairs(torch, stream, n):
    """n (start, stop) CUDA event pairs for the library's profiling hook.

    torch creates an event's handle lazily on its first record, so each pair
    is recorded once here; the library then re-records both around its main
    kernel, and elapsed_time reads those later records.
    """
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for a, b in pairs:
        a.record(stream)
        b.record(stream)
    return pairs


class Case:
    """One workload as the bench runs it: the timed step, its FLOP count, the
    dominant kernel the roofline describes, and the end-to-end variant that
    moves the step's inputs and results through pinned host memory."""


def make_conv_case(wan, torch, dev, w, rank, seed=0):
    """One causal Conv3d layer of the VAE on a chunk with its 2-frame cache, or
    (kind "time_down") one time-downsampling layer with its 1-frame cache."""
    B, T, H, W, ci, co = w.B, w.T, w.H, w.W, w.c_in, w.c_out
    down = w.kind == "time_down"
    gen = torch.Generator(device=dev)
    gen.manual_seed(input_seed(seed, rank))
    stream = torch.cuda.current_stream(dev)
    c = Case()
    c.stream = stream
    x = torch.randn(B, T, H, W, ci, device=dev, generator=gen).bfloat16()
    cache = torch.randn(B, 1 if down else 2, H, W, ci, device=dev, generator=gen).bfloat16()
    taps = (3,) if down else (3, 3, 3)
    wt = (torch.randn(co, *taps, ci, device=dev, generator=gen) / math.sqrt(w.taps() * ci)).bfloat16()
    bias = torch.randn(co, device=dev, generator=gen) * 0.1
    y = torch.empty(B, w.t_out(), H, W, co, dtype=torch.bfloat16, device=dev)
    cache_out = torch.empty_like(cache)
    entry = wan.wan_vae_time_downsample if down else wan.wan_vae_causal_conv3d

    def run():
        wan.check(entry(x, cache, wt, bias, y, cache_out, B, T, H, W, ci, co, stream))

    c.inputs, c.outputs = [x, cache, wt, bias], [y, cache_out]
    c.flops = c.kernel_flops = w.flops()
    c.kernel = "causal_conv3d_kernel<time_down>" if down else "causal_conv3d_kernel"
    c.launches, c.hbm_bytes, c.bound = 1, None, "tensor"

    def step(prof=None, rope_prof=None):
        if prof is not None:
            wan.check(wan.wan_profile_set_events(*prof))
        run()

    c.step = step
    c.in_bytes = sum(t.numel() * t.element_size() for t in c.inputs)
    c.out_bytes = sum(t.numel() * t.element_size() for t in c.outputs)
    return c


def input_seed(seed: int, rank: int) -> int:
    """torch generator seed of the bench inputs of (seed, rank)."""
    return 1000 * (seed + 1) + rank


def make_case(wan, torch, dev, w, rank, peaks, seed=0):
    if w.kind in CONV_KINDS:
        return make_conv_case(wan, torch, dev, w, rank, seed)
    B, L, H, d, grid = w.B, w.L, w.H, w.d, w.grid
    scale = 1.0 / math.sqrt(d)
    gen = torch.Generator(device=dev)
    gen.manual_seed(input_seed(seed, rank))
    stream = torch.cuda.current_stream(dev)
    c = Case()
    c.stream = stream
    fwd_flops = 4.0 * B * H * L * (w.Lk if w.kind == "cross_fwd" else L) * d
    if w.kind == "cross_fwd":
        from long_sequence_attention_02_b300 import synth

        Lk = w.Lk
        q = torch.randn(B, L, H, d, device=dev, generator=gen).bfloat16()
        k = torch.randn(B, Lk, H, d, device=dev, generator=gen).bfloat16()
        v = torch.randn(B, Lk, H, d, device=dev, generator=gen).bfloat16()
        lens_np = synth.kv_lens(0, B)
        lens = torch.from_numpy(lens_np).to(dev)
        o, lse = torch.empty_like(q), torch.empty(B, H, L, device=dev)

        def run():
            wan.check(wan.wan_xattn_fwd(q, k, v, lens, Lk, o, lse, B, grid, H, d, scale, stream))

        c.inputs, c.outputs = [q, k, v], [o, lse]
        c.flops, c.kernel, c.kernel_flops, c.launches = fwd_flops, "attn_fwd_kernel<false>", fwd_flops, 1
        c.extra_config = {"Lk": Lk, "kv_lens": lens_np.tolist(),
                          "useful_flop_per_step": 4.0 * H * L * d * float(lens_np.sum())}
        # HBM roofline: Q read + O written once, LSE written, K/V read once.
        c.hbm_bytes = q.numel() * 2 * 2 + lse.numel() * 4 + 2 * k.numel() * 2
        c.bound = "hbm"
    else:
        q = torch.randn(B, L, H, d, device=dev, generator=gen).bfloat16()
        k = torch.randn(B, L, H, d, device=dev, generator=gen).bfloat16()
        v = torch.randn(B, L, H, d, device=dev, generator=gen).bfloat16()
        o, lse = torch.empty_like(q), torch.empty(B, H, L, device=dev)
        tables = wan.rope_tables(grid, device=dev)
        wsf = wan.wan_attn_workspace_size(wan.WAN_OP_FWD, B, grid, H, d)
        if w.kind == "self_fwd":
            ws = torch.empty(wsf, dtype=torch.uint8, device=dev)

            def run():
                wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, grid, H, d, tables, scale, ws, wsf, stream))

            c.inputs, c.outputs = [q, k, v], [o, lse]
            c.flops, c.kernel, c.kernel_flops, c.launches = fwd_flops, "attn_fwd_kernel<true>", fwd_flops, 2
            c.hbm_bytes = None
            c.bound = "tensor"
            # the K rotation pre-pass: 256 B read + 256 B written per (token, head)
            c.rope_bytes = B * L * H * 512
        elif w.kind == "self_fwd_fp8":
            ws8 = wan.wan_attn_workspace_size(wan.WAN_OP_FWD_FP8, B, grid, H, d)
            ws = torch.empty(ws8, dtype=torch.uint8, device=dev)

            def run():
                wan.check(wan.wan_attn_fwd_fp8(q, k, v, o, lse, B, grid, H, d, tables, scale, ws, ws8, stream))

            c.inputs, c.outputs = [q, k, v], [o, lse]
            # amax pass, quantisation pass, attention
            c.flops, c.kernel, c.kernel_flops, c.launches = fwd_flops, "attn_fwd_fp8_kernel", fwd_flops, 3
            c.hbm_bytes = None
            c.bound = "tensor_fp8"
            c.dtype = "e4m3"
        else:  # forward + backward (one training step of the attention)
            do = torch.randn(B, L, H, d, device=dev, generator=gen).bfloat16()
            dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
            wsb = wan.wan_attn_workspace_size(wan.WAN_OP_BWD, B, grid, H, d)
            ws = torch.empty(max(wsf, wsb), dtype=torch.uint8, device=dev)
            pad = 1 if L % 128 else 0
            state = {"prof": None}

            def run():
                wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, grid, H, d, tables, scale, ws, wsf, stream))
                if state["prof"] is not None:
                    wan.check(wan.wan_profile_set_events(*state["prof"]))
                wan.check(wan.wan_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, grid, H, d, tables, scale, ws, wsb,
                                           stream))

            c.state = state
            c.inputs, c.outputs = [q, k, v, do], [dq, dk, dv]
            c.flops = 3.5 * fwd_flops
            c.kernel, c.kernel_flops = "attn_bwd_kernel", 2.5 * fwd_flops
            # forward: K rotation + attention; backward: Q and K rotation, row
            # pass (+ padding), attention backward, dQ rotation back
            c.launches = 2 + 5 + pad
            c.hbm_bytes = None
            c.bound = "tensor"

    def step(prof=None, rope_prof=None):
        if hasattr(c, "state"):
            c.state["prof"] = prof
        elif prof is not None:
            wan.check(wan.wan_profile_set_events(*prof))
        if rope_prof is not None and not hasattr(c, "state"):
            wan.check(wan.wan_profile_set_pass_events(wan.WAN_PASS_ROPE, *rope_prof))
        run()

    c.step = step
    c.in_bytes = sum(t.numel() * t.element_size() for t in c.inputs)
    c.out_bytes = sum(t.numel() * t.element_size() for t in c.outputs)
    return c


def read_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` recorded under profiles/ for this
    workload, or None if absent or taken from a different kernel source."""
    prof_path = os.path.join(HERE, "profiles", "traffic.json")
    try:
        with open(prof_path) as f:
            tr = json.load(f)
    except Exception:
        return None
    ent = tr.get(kernel, {})
    if ent.get("source_fingerprint") != source_fingerprint(kernel) or ent.get("workload") not in (None, workload):
        return None
    return ent.get("bytes_per_launch")


def run_ours(args, rank, world, local):
    import torch

    import long_sequence_attention_02_b300 as wan
    from long_sequence_attention_02_b300.workloads import CONV_WORKLOADS, WORKLOADS

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    peaks = _peaks()
    w = WORKLOADS[args.workload] if args.workload in WORKLOADS else CONV_WORKLOADS[args.workload]

    # One timed run per input seed; the line reports the median seed (by step
    # time) and lists all of them.
    runs = []
    for seed in args.seeds:
        c = make_case(wan, torch, dev, w, rank, peaks, seed)
        stream = c.stream
        for _ in range(args.warmup):
            c.step()
        torch.cuda.synchronize()
        wan.check(wan.wan_get_device_status())

        kev = timing_pairs(torch, stream, args.steps)
        rev = timing_pairs(torch, stream, args.steps) if getattr(c, "rope_bytes", None) else None
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(local)
        barrier(world)
        torch.cuda.synchronize()
        sampler.start()
        time.sleep(0.3)
        e0.record(stream)
        for i in range(args.steps):
            c.step(kev[i], rev[i] if rev else None)
        e1.record(stream)
        torch.cuda.synchronize()
        sampler.stop()
        barrier(world)
        wan.check(wan.wan_get_device_status())
        ms = e0.elapsed_time(e1) / args.steps
        runs.append({"seed": seed, "ms": ms, "ms_max": max_over_ranks(ms, world),
                     "kernel_ms": sum(a.elapsed_time(b) for a, b in kev) / args.steps,
                     "rope_ms": sum(a.elapsed_time(b) for a, b in rev) / args.steps if rev else None,
                     "sampler": sampler, "case": c})
    order = sorted(range(len(runs)), key=lambda r: runs[r]["ms_max"])
    med = runs[order[len(order) // 2]]
    for r in runs:
        if r is not med:
            r["case"] = None  # free the other seeds' buffers
    c, stream = med["case"], med["case"].stream
    ms_max, kernel_ms = med["ms_max"], med["kernel_ms"]
    clocks = ClockSampler.merge([r["sampler"] for r in runs])
    value = aggregate(c.flops, world, ms_max / 1e3) / 1e12

    # ----- end to end through the C ABI with host buffers
    # Every step uploads its inputs from pinned host memory, runs, and reads its
    # results back. Two device buffer sets let step i+1's upload and step i-1's
    # download (copy streams) overlap step i's compute, as a serving loop would;
    # each step's own copies stay inside the timed region, which runs from
    # before the first upload to the end of the last download.
    sets = [c, make_case(wan, torch, dev, w, rank, peaks, med["seed"])]
    hin = [t.cpu().pin_memory() for t in c.inputs]
    hout = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in c.outputs] for _ in sets]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(n_steps, start_event=None):
        comp_done, out_done = [None, None], [None, None]
        for i in range(n_steps):
            j = i & 1
            cs = sets[j]
            with torch.cuda.stream(s_in):
                if start_event is not None:
                    s_in.wait_event(start_event)
                if comp_done[j] is not None:  # the set's inputs are free once its last compute ended
                    s_in.wait_event(comp_done[j])
                for dst, src in zip(cs.inputs, hin):
                    dst.copy_(src, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            stream.wait_event(ev_in)
            if out_done[j] is not None:  # its outputs are free once read back
                stream.wait_event(out_done[j])
            cs.step()
            comp_done[j] = torch.cuda.Event()
            comp_done[j].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[j])
                for dst, src in zip(hout[j], cs.outputs):
                    dst.copy_(src, non_blocking=True)
                out_done[j] = torch.cuda.Event()
                out_done[j].record(s_out)
        for e in out_done:
            if e is not None:
                stream.wait_event(e)

    e2e_steps = max(2, min(args.steps, 10))
    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    e2e_run(e2e_steps, a0)
    a1.record(stream)
    torch.cuda.synchronize()
    wan.check(wan.wan_get_device_status())
    e2e_ms = max_over_ranks(a0.elapsed_time(a1) / e2e_steps, world)
    e2e = {"value": round(aggregate(c.flops, world, e2e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
           "h2d_bytes_per_step": c.in_bytes, "d2h_bytes_per_step": c.out_bytes, "ms_per_step": round(e2e_ms, 3),
           "steps": e2e_steps,
           "pipelining": "two device buffer sets; uploads and downloads on two copy streams overlap the "
                         "neighbouring steps' compute"}
    del hin, hout, sets

    also = {}
    if not args.no_extras and rank == 0:
        also = extras(wan, torch, dev, peaks, skip=w.name)

    traffic = read_traffic(c.kernel, w.name)
    sm_mhz, sm_max = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if c.bound == "tensor_fp8":
        # fp8 dense peak: the measured bf16 GEMM burst peak x the nominal fp8/bf16 ratio (4.5 / 2.25 PF)
        peak = 2.0 * peaks["bf16_tflops"]
        achieved = c.kernel_flops / (kernel_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": c.kernel, "achieved": round(achieved, 2), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "peak_kind": f"fp8 = 2 x bf16 burst ({peaks['source']}; nominal 4.5 / 2.25 PF)",
                    "frac_of_2x_bf16_sustained": round(achieved / (2.0 * peaks["bf16_tflops_sustained"]), 4),
                    "frac_of_4.5PF_fp8_spec": round(achieved / 4500.0, 4),
                    "kernel_ms": round(kernel_ms, 3), "traffic": traffic}
    elif c.bound == "tensor":
        peak = peaks["bf16_tflops"]
        achieved = c.kernel_flops / (kernel_ms / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": c.kernel, "achieved": round(achieved, 2), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "peak_kind": f"bf16 GEMM burst ({peaks['source']})",
                    "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
                    "frac_of_2.25PF_spec": round(achieved / 2250.0, 4),
                    "kernel_ms": round(kernel_ms, 3), "traffic": traffic}
    else:
        peak = peaks["hbm_gbs"]
        achieved = c.hbm_bytes / (kernel_ms / 1e3) / 1e9
        roofline = {"bound": "hbm", "kernel": c.kernel, "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "peak_kind": f"HBM copy ({peaks['source']})",
                    "algorithmic_bytes": c.hbm_bytes, "kernel_ms": round(kernel_ms, 3), "traffic": traffic,
                    "tensor_tflops_nominal": round(c.kernel_flops / (kernel_ms / 1e3) / 1e12, 2)}
    if sm_mhz:
        # time x clock: the kernel's cycle count in millions, comparable across clocks
        roofline["kernel_ms_x_median_sm_mhz"] = round(kernel_ms * sm_mhz, 1)
        if c.bound != "hbm" and sm_max:
            roofline["achieved_if_at_max_sm_clock"] = round(achieved * sm_max / sm_mhz, 1)
    hbm_phases = {}
    if med["rope_ms"]:
        gbs = c.rope_bytes / (med["rope_ms"] / 1e3) / 1e9
        hbm_phases["rope_rotate_kernel"] = {"pass": f"K rotation of {w.name} ({w.L} x {w.H})",
                                            "ms": round(med["rope_ms"], 4), "bytes": c.rope_bytes,
                                            "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4)}
    if w.kind in CONV_KINDS:
        down = w.kind == "time_down"
        x_mib = c.inputs[0].numel() * 2 / 2**20
        config = {"workload": w.name, "kind": w.kind, "B": w.B, "frames": w.T, "height": w.H, "width": w.W,
                  "c_in": w.c_in, "c_out": w.c_out, "kernel": [3, 1, 1] if down else [3, 3, 3],
                  "cache": f"{1 if down else 2} frame(s) of the previous chunk, written for the next one",
                  "flop_per_step": c.flops,
                  "l2": (f"input x {x_mib:.0f} MiB > L2 126 MB (no flush needed)" if x_mib * 2**20 > 126e6 else
                         f"input x {x_mib:.0f} MiB fits L2 126 MB (not flushed)"),
                  "frac_of_2.25PF_spec": round(value / 2250.0, 4)}
    else:
        config = {"workload": w.name, "kind": w.kind, "B": w.B, "grid": list(w.grid), "tokens": w.L, "heads": w.H,
                  "head_dim": w.d, "flop_per_step": c.flops,
                  "l2": f"inputs {c.in_bytes / 2**30:.2f} GiB > L2 126 MB (no flush needed)",
                  "frac_of_2.25PF_spec": round(value / 2250.0, 4)}
    if w.kind not in ("cross_fwd",) + CONV_KINDS:
        config["theta"] = 10000.0
    config.update(getattr(c, "extra_config", {}))
    line = {
        "metric": CONV_METRIC if w.kind in CONV_KINDS else METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": getattr(c, "dtype", "bf16"),
        "data": (f"synthetic: bf16 N(0,1) activations and cache, N(0,1)/sqrt({w.taps()} C_in) weights (torch "
                 "generator, seed 1000*(s+1)+rank for input seeds s)" if w.kind in CONV_KINDS else
                 "synthetic: bf16 N(0,1) inputs (torch generator, seed 1000*(s+1)+rank for input seeds s)"),
        "config": config,
        "roofline": roofline,
        "clocks": clocks,
        "e2e": e2e,
        "gpu_launches": c.launches * args.steps * len(runs),
        "seeds": {str(r["seed"]): round(r["ms_max"], 3) for r in runs},
        "median_seed": med["seed"],
    }
    if also:
        hbm_phases.update(also.pop("hbm_phases", {}))
        line["also"] = also
    if hbm_phases:
        line["hbm_phases"] = hbm_phases
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_rows)
    if rank == 0:
        print(json.dumps(line), flush=True)


def extras(wan, torch, dev, peaks, skip=None):
    """Secondary workloads, each timed with CUDA events (3 iterations after 2 warm-ups)."""
    from long_sequence_attention_02_b300.workloads import WORKLOADS

    out = {}
    stream = torch.cuda.current_stream(dev)

    def timeit(fn, iters=3, warm=2, prof=False):
        for _ in range(warm):
            fn(None)
        torch.cuda.synchronize()
        ev = timing_pairs(torch, stream, iters)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(iters):
            fn(ev[i] if prof else None)
        b.record(stream)
        torch.cuda.synchronize()
        wan.check(wan.wan_get_device_status())
        tot = a.elapsed_time(b) / iters
        ker = sum(x.elapsed_time(y) for x, y in ev) / iters if prof else None
        return tot, ker

    _extra_tiny(wan, torch, dev, WORKLOADS["tiny_3x8x8_h2"], stream, out)
    # 480p self-attention forward
    w = WORKLOADS["wan1.3b_480p_self_fwd"]
    if w.name == skip:
        w = None
    if w is not None:
        _extra_480p(wan, torch, dev, w, stream, timeit, out)
    w = WORKLOADS["wan14b_720p_cross_fwd"]
    if w.name != skip:
        _extra_cross(wan, torch, dev, w, stream, timeit, out, peaks)
    w = WORKLOADS["train_64x64x64_fwd_bwd"]
    if w.name != skip:
        _extra_train(wan, torch, dev, w, stream, timeit, out)
    from long_sequence_attention_02_b300.workloads import CONV_WORKLOADS

    w = CONV_WORKLOADS["wan_vae_conv3d_360x640_192"]
    if w.name != skip:
        _extra_conv(wan, torch, dev, w, stream, timeit, out, peaks)
    w = CONV_WORKLOADS["wan_vae_time_down_180x320_192"]
    if w.name != skip:
        _extra_conv(wan, torch, dev, w, stream, timeit, out, peaks)
    w = WORKLOADS["wan14b_720p_self_fwd_fp8"]
    if w.name != skip:
        _extra_fp8(wan, torch, dev, w, stream, timeit, out, peaks)
    _extra_dual(wan, torch, dev, WORKLOADS["wan14b_720p_cross_fwd"], stream, timeit, out, peaks)
    _extra_ring(wan, torch, dev, WORKLOADS["wan14b_720p_self_fwd"], stream, timeit, out, peaks)
    return out


def _extra_fp8(wan, torch, dev, w, stream, timeit, out, peaks):
    """FP8 forward of the 75,600-token, 40-head problem: the whole call (amax,
    quantisation, attention) and its attention kernel."""
    B, L, H, d = w.B, w.L, w.H, w.d
    q = torch.randn(B, L, H, d, device=dev).bfloat16()
    k, v = torch.randn_like(q), torch.randn_like(q)
    o, lse = torch.empty_like(q), torch.empty(B, H, L, device=dev)
    tab = wan.rope_tables(w.grid, device=dev)
    wsb = wan.wan_attn_workspace_size(wan.WAN_OP_FWD_FP8, B, w.grid, H, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def f(p):
        if p is not None:
            wan.wan_profile_set_events(*p)
        wan.check(wan.wan_attn_fwd_fp8(q, k, v, o, lse, B, w.grid, H, d, tab, 1 / math.sqrt(d), ws, wsb, stream))

    tot, ker = timeit(f, iters=3, prof=True)
    fl = 4.0 * B * H * L * L * d
    out[w.name] = {"ms": round(tot, 3), "tflops": round(fl / tot / 1e9, 1), "kernel_tflops": round(fl / ker / 1e9, 1),
                   "kernel_frac_of_fp8_peak": round(fl / ker / 1e9 / (2 * peaks["bf16_tflops"]), 4),
                   "peak": "fp8 = 2 x the measured bf16 burst (nominal 4.5 / 2.25 PF)"}
    del q, k, v, o, lse, ws


def _extra_dual(wan, torch, dev, w, stream, timeit, out, peaks):
    """Decoupled text + image cross-attention of image-to-video models on the
    720p cross-attention shape: 512 text keys (seeded lengths) and 257 image
    keys (a CLIP ViT-H/14 embedding of 16 x 16 patches + 1; the pages give no
    count). Two launches; the second adds its result to the first's O."""
    from long_sequence_attention_02_b300 import synth

    B, Lq, H, d, Lk = w.B, w.L, w.H, w.d, w.Lk
    Li = 257
    q = torch.randn(B, Lq, H, d, device=dev).bfloat16()
    kt, vt = torch.randn(B, Lk, H, d, device=dev).bfloat16(), torch.randn(B, Lk, H, d, device=dev).bfloat16()
    ki, vi = torch.randn(B, Li, H, d, device=dev).bfloat16(), torch.randn(B, Li, H, d, device=dev).bfloat16()
    lens_np = synth.kv_lens(0, B)
    lens = torch.from_numpy(lens_np).to(dev)
    o, lse = torch.empty_like(q), torch.empty(B, H, Lq, device=dev)

    def f(p):
        wan.check(wan.wan_xattn_fwd_dual(q, kt, vt, lens, Lk, ki, vi, None, Li, o, lse, B, w.grid, H, d,
                                          1 / math.sqrt(d), stream))

    tot, _ = timeit(f, iters=10)
    qb = q.numel() * 2
    moved = 5 * qb + lse.numel() * 4 + 2 * (kt.numel() + ki.numel()) * 2  # Q twice, O written twice, read once
    floor = 2 * qb + lse.numel() * 4 + 2 * (kt.numel() + ki.numel()) * 2  # Q read and O written once
    out["wan14b_720p_xattn_dual_txt512_img257"] = {
        "ms": round(tot, 3), "tflops_nominal": round(4.0 * B * H * Lq * (Lk + Li) * d / tot / 1e9, 1),
        "kv_lens_txt": lens_np.tolist(), "image_keys": Li, "bytes_moved": moved,
        "gbs": round(moved / tot / 1e6, 1), "hbm_frac": round(moved / tot / 1e6 / peaks["hbm_gbs"], 3),
        "single_pass_floor_ms": round(floor / peaks["hbm_gbs"] / 1e6, 3)}
    del q, kt, vt, ki, vi, o, lse


def _extra_ring(wan, torch, dev, w, stream, timeit, out, peaks):
    """The 75,600-token, 40-head forward as two Ring steps over the K/V halves
    (the second merges into the first's O and LSE by log-sum-exp), against the
    one-call forward's FLOP."""
    B, L, H, d = w.B, w.L, w.H, w.d
    q = torch.randn(B, L, H, d, device=dev).bfloat16()
    k, v = torch.randn_like(q), torch.randn_like(q)
    o, lse = torch.empty_like(q), torch.empty(B, H, L, device=dev)
    tab = wan.rope_tables(w.grid, device=dev)
    wsb = wan.wan_attn_workspace_size(wan.WAN_OP_FWD, B, w.grid, H, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
    half = L // 2
    chunks = [(0, half), (half, L - half)]
    kc = [k[:, a:a + n].contiguous() for a, n in chunks]
    vc = [v[:, a:a + n].contiguous() for a, n in chunks]

    def f(p):
        for i, (a, n) in enumerate(chunks):
            wan.check(wan.wan_attn_fwd_ring_step(q, kc[i], vc[i], o, lse, B, w.grid, H, d, tab, 1 / math.sqrt(d), 0,
                                                 L, a, n, 1 if i else 0, ws, wsb, stream))

    tot, _ = timeit(f, iters=3)
    fl = 4.0 * B * H * L * L * d
    out["wan14b_720p_self_fwd_ring2"] = {"ms": round(tot, 3), "tflops": round(fl / tot / 1e9, 1),
                                         "steps": 2, "kv_chunk_tokens": half}
    del q, k, v, o, lse, ws, kc, vc


def _extra_tiny(wan, torch, dev, w, stream, out, iters=200):
    """Latency of the tiny forward (192 tokens, 2 heads): a wan_attn_fwd call
    (K rotation + attention) and its attention kernel alone, in microseconds."""
    B, L, H, d = w.B, w.L, w.H, w.d
    q = torch.randn(B, L, H, d, device=dev).bfloat16()
    k, v = torch.randn_like(q), torch.randn_like(q)
    o, lse = torch.empty_like(q), torch.empty(B, H, L, device=dev)
    tab = wan.rope_tables(w.grid, device=dev)
    wsb = wan.wan_attn_workspace_size(0, B, w.grid, H, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def call():
        wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, w.grid, H, d, tab, 1 / math.sqrt(d), ws, wsb, stream))

    for _ in range(20):
        call()
    torch.cuda.synchronize()
    ev = timing_pairs(torch, stream, iters)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(iters):
        wan.wan_profile_set_events(*ev[i])
        call()
    b.record(stream)
    torch.cuda.synchronize()
    wan.check(wan.wan_get_device_status())
    us = a.elapsed_time(b) / iters * 1e3
    ker = statistics.median(x.elapsed_time(y) for x, y in ev) * 1e3
    out[w.name] = {"us_per_call": round(us, 2), "kernel_us_median": round(ker, 2),
                   "note": "back-to-back calls on one stream; latency-bound (192 tokens)"}
    # The same call captured once in a CUDA graph and replayed: the device
    # latency of the two kernels without the host's per-call work between them.
    try:
        def call_current():
            wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, w.grid, H, d, tab, 1 / math.sqrt(d), ws, wsb))

        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                call_current()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call_current()
        for _ in range(20):
            graph.replay()
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(iters):
            graph.replay()
        b.record(stream)
        torch.cuda.synchronize()
        wan.check(wan.wan_get_device_status())
        out[w.name]["graph_us_per_call"] = round(a.elapsed_time(b) / iters * 1e3, 2)
    except Exception as e:  # report, do not fail the bench line
        out[w.name]["graph_us_per_call"] = None
        out[w.name]["graph_error"] = str(e)[:200]


def _extra_480p(wan, torch, dev, w, stream, timeit, out):
    B, L, H, d = w.B, w.L, w.H, w.d
    q = torch.randn(B, L, H, d, device=dev).bfloat16()
    k, v = torch.randn_like(q), torch.randn_like(q)
    o, lse = torch.empty_like(q), torch.empty(B, H, L, device=dev)
    tab = wan.rope_tables(w.grid, device=dev)
    wsb = wan.wan_attn_workspace_size(0, B, w.grid, H, d)
    ws = torch.empty(wsb, dtype=torch.uint8, device=dev)

    def f480(p):
        if p is not None:
            wan.wan_profile_set_events(*p)
        wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, w.grid, H, d, tab, 1 / math.sqrt(d), ws, wsb, stream))

    tot, ker = timeit(f480, iters=10, prof=True)
    fl = 4.0 * B * H * L * L * d
    out[w.name] = {"ms": round(tot, 3), "tflops": round(fl / tot / 1e9, 1), "kernel_tflops": round(fl / ker / 1e9, 1)}
    del q, k, v, o, lse, ws


def _extra_cross(wan, torch, dev, w, stream, timeit, out, peaks):
    B, Lq, H, d, Lk = w.B, w.L, w.H, w.d, w.Lk
    q = torch.randn(B, Lq, H, d, device=dev).bfloat16()
    k = torch.randn(B, Lk, H, d, device=dev).bfloat16()
    v = torch.randn_like(k)
    from long_sequence_attention_02_b300 import synth

    lens_np = synth.kv_lens(0, B)
    lens = torch.from_numpy(lens_np).to(dev)
    o, lse = torch.empty_like(q), torch.empty(B, H, Lq, device=dev)

    def fx(p):
        if p is not None:
            wan.wan_profile_set_events(*p)
        wan.check(wan.wan_xattn_fwd(q, k, v, lens, Lk, o, lse, B, w.grid, H, d, 1 / math.sqrt(d), stream))

    tot, _ = timeit(fx, iters=10)
    nominal = 4.0 * B * H * Lq * Lk * d
    useful = 4.0 * H * Lq * d * float(lens_np.sum())
    hbm = (q.numel() * 2 * 2 + lse.numel() * 4 + k.numel() * 2 * 2)
    out[w.name] = {"ms": round(tot, 3), "tflops_nominal": round(nominal / tot / 1e9, 1),
                   "tflops_useful": round(useful / tot / 1e9, 1), "kv_lens": lens_np.tolist(),
                   "gbs": round(hbm / tot / 1e6, 1), "hbm_frac": round(hbm / tot / 1e6 / peaks["hbm_gbs"], 3)}
    del q, k, v, o, lse


def _extra_train(wan, torch, dev, w, stream, timeit, out):
    B, L, H, d = w.B, w.L, w.H, w.d
    q = torch.randn(B, L, H, d, device=dev).bfloat16()
    k, v, do = torch.randn_like(q), torch.randn_like(q), torch.randn_like(q)
    o, lse = torch.empty_like(q), torch.empty(B, H, L, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    tab = wan.rope_tables(w.grid, device=dev)
    wsf = wan.wan_attn_workspace_size(0, B, w.grid, H, d)
    wsb = wan.wan_attn_workspace_size(1, B, w.grid, H, d)
    ws = torch.empty(max(wsf, wsb), dtype=torch.uint8, device=dev)
    sc = 1 / math.sqrt(d)

    passes = {n: timing_pairs(torch, stream, 2) for n in ("rows", "post")}
    calls = {"n": 0}

    def ftrain(p):
        wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, w.grid, H, d, tab, sc, ws, wsf, stream))
        if p is not None:
            wan.wan_profile_set_events(*p)
            i = calls["n"]
            calls["n"] += 1
            wan.check(wan.wan_profile_set_pass_events(wan.WAN_PASS_ROWS, *passes["rows"][i]))
            wan.check(wan.wan_profile_set_pass_events(wan.WAN_PASS_POST, *passes["post"][i]))
        wan.check(wan.wan_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, B, w.grid, H, d, tab, sc, ws, wsb, stream))

    def ffwd(p):
        if p is not None:
            wan.wan_profile_set_events(*p)
        wan.check(wan.wan_attn_fwd(q, k, v, o, lse, B, w.grid, H, d, tab, sc, ws, wsf, stream))

    ffl = 4.0 * B * H * L * L * d
    tot_f, ker_f = timeit(ffwd, iters=2, warm=1, prof=True)
    tot, ker_b = timeit(ftrain, iters=2, warm=1, prof=True)
    out[w.name] = {"ms_fwd": round(tot_f, 2), "ms_fwd_bwd": round(tot, 2),
                   "tflops_fwd": round(ffl / tot_f / 1e9, 1),
                   "tflops_bwd_kernel": round(2.5 * ffl / ker_b / 1e9, 1),
                   "tflops_bwd": round(2.5 * ffl / (tot - tot_f) / 1e9, 1),
                   "tflops_step": round(3.5 * ffl / tot / 1e9, 1)}
    # HBM passes of the backward: bytes per (token, head) from what each reads and writes
    n = B * L * H
    phases = out.setdefault("hbm_phases", {})
    for kname, key, per, what in (
            ("bwd_rows_kernel", "rows", 512 + 4 + 8, "D = rowsum(dO * O) and LSE * log2 e: O, dO, LSE read; 2 floats written"),
            ("rope_unrotate_f32_kernel", "post", 512 + 256, "dQ = R^T dQ_acc: fp32 read, bf16 written")):
        ms = sum(a.elapsed_time(b) for a, b in passes[key][:calls["n"]]) / max(1, calls["n"])
        gbs = n * per / (ms / 1e3) / 1e9
        phases[kname] = {"pass": f"{what} ({w.name}, {L} x {H})", "ms": round(ms, 4), "bytes": n * per,
                         "gbs": round(gbs, 1), "frac_of_hbm": round(gbs / _peaks()["hbm_gbs"], 4)}


def _extra_conv(wan, torch, dev, w, stream, timeit, out, peaks):
    c = make_conv_case(wan, torch, dev, w, 0)
    tot, ker = timeit(lambda p: c.step(p), iters=5, prof=True)
    out[w.name] = {"ms": round(tot, 3), "tflops": round(w.flops() / tot / 1e9, 1),
                   "kernel_tflops": round(w.flops() / ker / 1e9, 1),
                   "kernel_frac_of_bf16_sustained": round(w.flops() / ker / 1e9 / peaks["bf16_tflops_sustained"], 4)}
    if w.kind == "time_down":
        # Compulsory bytes of the kernel: x and the cache read once, y written once, the weights.
        io = (w.B * (w.T + 1) * w.H * w.W * w.c_in + w.B * w.t_out() * w.H * w.W * w.c_out
              + 3 * w.c_in * w.c_out) * 2
        out[w.name].update({"kernel_bytes": io, "kernel_gbs": round(io / ker / 1e6, 1),
                            "kernel_frac_of_hbm": round(io / ker / 1e6 / peaks["hbm_gbs"], 4),
                            "note": "inputs (89 MB) fit L2; between HBM and tensor bound"})
    del c


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)


KERNEL_SOURCES = {
    "attn_fwd_kernel<true>": ("attn_fwd.cu", "common.cuh"),
    "attn_fwd_kernel<false>": ("attn_fwd.cu", "common.cuh"),
    "attn_bwd_kernel": ("attn_bwd.cu", "common.cuh"),
    "attn_fwd_fp8_kernel": ("attn_fwd_fp8.cu", "common.cuh"),
    "causal_conv3d_kernel": ("conv3d.cu", "common.cuh"),
    "causal_conv3d_kernel<time_down>": ("conv3d.cu", "common.cuh"),
}


def source_fingerprint(kernel: str = "attn_fwd_kernel<true>") -> str:
    import hashlib

    h = hashlib.sha1()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(HERE, "long_sequence_attention_02_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def _oracle_rows(w, rows_per_head: int, heads: int, seed: int = 0):
    """Time the oracle on `rows_per_head` query rows of `heads` heads.

    Self-attention rows run the oracle's 3D-RoPE forward (and, for a training
    workload, its dQ backward too); cross-attention rows attend to the valid
    text keys of batch 0. Returns (rows, seconds, convention FLOP per row).
    """
    import numpy as np

    from long_sequence_attention_02_b300 import synth
    from oracle import ref

    L, d, H = w.L, w.d, w.H
    Lk = w.Lk if w.kind == "cross_fwd" else L
    t0 = time.perf_counter()
    n = 0
    for h in range(heads):
        idx_k = (np.arange(Lk, dtype=np.uint64)[:, None] * H + h) * d + np.arange(d, dtype=np.uint64)[None, :]
        kh = synth.bf16_bits_to_f64(synth.normal_bf16_at(seed, synth.STREAM_K, idx_k))
        vh = synth.bf16_bits_to_f64(synth.normal_bf16_at(seed, synth.STREAM_V, idx_k))
        rows = np.arange(rows_per_head, dtype=np.int64) * (L // rows_per_head)
        idx_q = (rows.astype(np.uint64)[:, None] * H + h) * d + np.arange(d, dtype=np.uint64)[None, :]
        qr = synth.bf16_bits_to_f64(synth.normal_bf16_at(seed, synth.STREAM_Q, idx_q))
        if w.kind == "cross_fwd":
            ref.softmax_attention(qr, kh, vh, 1.0 / math.sqrt(d), int(synth.kv_lens(seed, w.B)[0]))
        else:
            ref.self_attention_fwd_rows(qr, rows, kh, vh, w.grid)
            if w.kind == "self_fwd_bwd":
                dor = synth.bf16_bits_to_f64(synth.normal_bf16_at(seed, synth.STREAM_DO, idx_q))
                ref.self_attention_bwd_dq_rows(qr, dor, rows, kh, vh, w.grid)
        n += rows_per_head
    dt = time.perf_counter() - t0
    per_row = 4.0 * Lk * d * (3.5 if w.kind == "self_fwd_bwd" else 1.0)
    return n, dt, per_row


def _oracle_conv(w, n_pos: int, seed: int = 0):
    """Time the conv oracle on n_pos output positions, each computed from its
    3 x 3 x 3 window (3 x 1 x 1 for the time-downsampling layer: one cached
    frame and two chunk frames), drawn from the seeded generator, against all
    C_out. Returns (positions, seconds, FLOP per position)."""
    import numpy as np

    from long_sequence_attention_02_b300 import synth
    from oracle import vae

    ci, co, taps = w.c_in, w.c_out, w.taps()
    shape = (co, 3, ci) if w.kind == "time_down" else (co, 3, 3, 3, ci)
    wt = synth.bf16_bits_to_f64(synth.normal_bf16(seed, synth.STREAM_V, shape)) / math.sqrt(taps * ci)
    rng = np.random.default_rng(seed)
    t0 = time.perf_counter()
    for i in range(n_pos):
        off = int(rng.integers(0, 2**40)) * taps * ci
        if w.kind == "time_down":
            win = synth.bf16_bits_to_f64(synth.normal_bf16(seed, synth.STREAM_Q, (1, 3, 1, 1, ci), offset=off))
            vae.causal_time_downsample(win[:, 1:], wt, None, win[:, :1])
        else:
            win = synth.bf16_bits_to_f64(synth.normal_bf16(seed, synth.STREAM_Q, (1, 3, 3, 3, ci), offset=off))
            vae.causal_conv3d_at(win, wt, None, None, [(0, 2, 1, 1)])
    dt = time.perf_counter() - t0
    return n_pos, dt, 2.0 * taps * ci * co


def cpu_baseline(w, rows_per_head: int):
    if w.kind in CONV_KINDS:
        n, dt, per = _oracle_conv(w, 2 * rows_per_head)
        win = "3x1x1" if w.kind == "time_down" else "3x3x3"
        return {"value": round(per * n / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                "sample": f"{n} output positions of {w.name}, each from its {win} window against all {w.c_out} "
                          f"output channels, fp64 numpy, {dt:.1f} s", "positions_per_s": round(n / dt, 1)}
    n, dt, per_row = _oracle_rows(w, rows_per_head, heads=2)
    what = {"self_fwd": "forward", "self_fwd_fp8": "forward", "cross_fwd": "cross-attention forward",
            "self_fwd_bwd": "forward + dQ backward"}[w.kind]
    return {"value": round(per_row * n / dt / 1e12, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} query rows (2 heads x {rows_per_head}) of {w.name}, oracle {what} against all keys, "
                      f"fp64 numpy, {dt:.1f} s", "rows_per_s": round(n / dt, 1)}


def run_reference(args, rank, world):
    from long_sequence_attention_02_b300.workloads import WORKLOADS

    if rank != 0:
        return
    if args.workload not in WORKLOADS:
        return run_reference_conv(args, world)
    w = WORKLOADS[args.workload]
    rows = args.ref_rows
    for _ in range(args.warmup):
        _oracle_rows(w, rows, heads=1)
    times, n_tot, per_row = [], 0, 0.0
    for _ in range(args.steps):
        n, dt, per_row = _oracle_rows(w, rows, heads=1)
        times.append(dt)
        n_tot += n
    dt = sum(times)
    fl = per_row * n_tot
    value = fl / dt / 1e12
    sample = f"{rows} query rows of one head per step against all keys (fp64 numpy oracle)"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: bf16 N(0,1) from the seeded SplitMix64 generator",
        "config": {"workload": w.name, "B": w.B, "grid": list(w.grid), "tokens": w.L, "heads": w.H,
                   "head_dim": w.d},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_conv(args, world):
    from long_sequence_attention_02_b300.workloads import CONV_WORKLOADS

    w = CONV_WORKLOADS[args.workload]
    n = 4 * args.ref_rows
    for _ in range(args.warmup):
        _oracle_conv(w, n)
    dt, fl = 0.0, 0.0
    for _ in range(args.steps):
        k, t, per = _oracle_conv(w, n)
        dt += t
        fl += per * k
    value = fl / dt / 1e12
    line = {
        "impl": "reference", "metric": CONV_METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: bf16 N(0,1) from the seeded SplitMix64 generator",
        "config": {"workload": w.name, "kind": w.kind, "B": w.B, "frames": w.T, "height": w.H, "width": w.W,
                   "c_in": w.c_in, "c_out": w.c_out},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": f"{n} output positions per step, each from its "
                                   f"{'3x1x1' if w.kind == 'time_down' else '3x3x3'} window (fp64 numpy oracle)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="wan14b_720p_self_fwd")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=512)
    ap.add_argument("--ref-rows", type=int, default=64)
    ap.add_argument("--seeds", type=int, nargs="+", default=[0, 1, 2],
                    help="input seeds; each is timed and the median seed is reported")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup(args.gpus, gpu=args.impl != "reference")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()

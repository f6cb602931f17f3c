#!/usr/bin/env python
"""Throughput of the routed expert-FFN layer on B300.

Headline workload (one JSON line on stdout, rank 0):
  decode  -- one token (B=1) through a stack of 48 resident MoE layers
             (H=2048, E=512, I=512, top-10, 2-bit block-32 weights, residual
             add between layers); `value` is per-layer tokens/s, i.e. tokens
             through one layer per second, measured over the whole stack so
             every step reads 48 distinct layers' experts (~673 MB > L2).
Further objects of the same line:
  decode_t8 -- the same stack at 8 tokens per call (a multi-token decode call)
  prefill   -- a 4,096-token chunk through one layer whose router bias is
               Zipf-skewed (some experts get no token; inputs 0.57 GB > L2)
  stack     -- a 32,768-token prompt as 8 chunks of 4,096 tokens through all
               48 layers, then 256 decode steps of one token
  bits3     -- 3-bit weights: a 64-token verify window and a 16,384-token chunk
  mode_sweep-- GEMV vs grouped-GEMM expert path per call size
All are replayed from CUDA graphs of the library's C-ABI calls.  Roofline
fractions use MEASURED_PEAKS.json.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the fp64 reference this library is
checked against) on the host cores on a bounded sample of the decode
workload.  Under torchrun every rank runs its own replica (weak scaling, no
collective on the data path); timings are reduced by MAX over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE expert-FFN tokens/s (4K prefill, B=1 decode); % of int8 / HBM roofline"
H, I, E, K_TOP = 2048, 512, 512, 10
N_LAYERS = 48
DECODE_T = 1
DECODE_T8 = 8
PREFILL_T = 4096
PROMPT_T = 32768  # the stack's prompt, read in PREFILL_T-token chunks
STACK_DECODE_STEPS = 256
EXPERT_BYTES = 3 * I * (H // 32) * (8 + 2)  # 2-bit codes + fp16 scales of gate, up, down = 983,040
EXPERT_BYTES3 = 3 * I * (H // 32) * (12 + 2)  # 3-bit: 1,376,256
ROUTER_BYTES = E * H * 4  # fp32 router matrix, read once per decode call
VERIFY_T = 64  # 3-bit decode: a multi-token verify window
PREFILL3_T = 16384  # 3-bit prefill chunk, uniform routing
SWEEP_T = (8, 16, 32, 64, 128, 256, 512, 1024)  # token counts of the GEMV / grouped-GEMM crossover sweep
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# current kernel versions from one ncu --set full capture (profiles/), with
# its source; set to None when a kernel changes until it is captured again
DECODE_LAYER_TRAFFIC = dict(bytes=4.220416e6 + 9.925376e6,
                            source=("ncu: route_gemv_kernel 4.22 MB + ffn_gemv_kernel 9.93 MB, one B=1 layer "
                                    "(profiles/route_gemv_decode_T1.md, ffn_gemv_decode_T1.md)"))
GEMM_GU_TRAFFIC = dict(bytes=688.752384e6 + 20.226048e6,
                       source="ncu: ffn_gemm_kernel<1,2> 688.8 MB read + 20.2 MB written (profiles/ffn_gemm_gateup_prefill_4k.md)")


# ------------------------------------------------------------------ helpers


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sus=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    except (OSError, KeyError, ValueError):
        return dict(hbm=6400.0, bf16=1800.0, bf16_sus=1400.0, source="fallback")


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def reduce_max(v: float, world: int) -> float:
    """Max over ranks (the slowest replica sets the job's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, seconds: float, world: int) -> dict:
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    t = reduce_max(seconds, world)
    return dict(value=units_per_rank * world / t, seconds=t)


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moeq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()
            self.fh.close()

    def summary(self):
        if not self.proc:
            return None
        sms, maxs, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sms.append(float(parts[1]))
                    maxs.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sms:
            return None
        return dict(sm_mhz=statistics.median(sms), sm_max_mhz=max(maxs), samples=len(sms), reasons=sorted(reasons))


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------ oracle (CPU)


def oracle_decode_rate(layer_np, n_tokens: int, seed: int = 3):
    """Oracle layer-tokens/s on the host cores for n_tokens independent tokens."""
    import oracle
    import synth

    x = synth.make_x(n_tokens, H, seed=seed).numpy()
    threads = cpu_cores()
    t0 = time.perf_counter()
    oracle.layer(x, *layer_np, 2, K_TOP, residual=True, nthreads=threads)
    dt = time.perf_counter() - t0
    return n_tokens / dt, threads, dt


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch

    import synth

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    layer = synth.make_layer(synth.FULL, seed=0, layer=0, device=dev)
    lnp = layer.numpy()
    del layer
    n_tok = max(1, args.ref_tokens)
    for _ in range(args.warmup):
        oracle_decode_rate(lnp, n_tok)
    rates, secs, threads = [], [], 1
    for _ in range(args.steps):
        r, threads, dt = oracle_decode_rate(lnp, n_tok)
        rates.append(r)
        secs.append(dt)
    value = n_tok * args.steps / sum(secs)
    sample = (f"{n_tok} independent decode tokens through one 2048/512/512 top-10 2-bit layer per step "
              f"(each token is one B=1 decode call; the stack's other layers are identical work)")
    print(json.dumps(dict(
        impl="reference", metric=METRIC, value=value, unit="tokens/s", n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=1e3 * sum(secs) / args.steps, higher_is_better=True, scaling="weak",
        vs_baseline=None, dtype="f64", data="synthetic",
        config=dict(workload="decode: B=1 tokens through a 2048/512/512 top-10 2-bit MoE layer (CPU oracle)",
                    T=DECODE_T, layers_sampled=1),
        cpu_baseline=dict(value=value, unit="tokens/s", cores=threads, kind="oracle", sample=sample),
        e2e=dict(value=value, unit="tokens/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))), flush=True)


# ------------------------------------------------------------ ours (GPU)


class Gpu:
    """Device, library, peaks and the timing helpers shared by the sections."""

    def __init__(self, world, local):
        import torch

        import quantized_mixture_experts_token_b300 as moeq

        self.torch, self.moeq, self.world = torch, moeq, world
        self.dev = torch.device("cuda", local)
        self.pk = peaks()

    def barrier(self):
        if self.world > 1:
            import torch.distributed as dist

            dist.barrier()

    def timed(self, fn, steps, warmup):
        """Seconds for `steps` calls of fn after `warmup` untimed ones (CUDA events)."""
        torch = self.torch
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        self.barrier()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        self.barrier()
        return s.elapsed_time(e) / 1e3

    def graph(self, fn):
        torch = self.torch
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g


class Pipelined:
    """Chunks through double-buffered graphs with the host copies on their own
    streams: the upload of chunk c (pinned host -> device buffer c % 2) waits
    until chunk c - 2 has computed, the compute of chunk c waits for its upload
    and for the download of chunk c - 2 (the same output buffer), and the
    download of chunk c waits for its compute."""

    def __init__(self, gpu, graphs, dev_in, dev_out, host_in, host_out):
        torch = gpu.torch
        self.gpu, self.graphs, self.dev_in, self.dev_out = gpu, graphs, dev_in, dev_out
        self.host_in, self.host_out = host_in, host_out
        self.up, self.down = torch.cuda.Stream(gpu.dev), torch.cuda.Stream(gpu.dev)
        self.ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("up", "comp", "down")}
        self.started = [False, False]

    def chunk(self, c):
        torch = self.gpu.torch
        b, comp = c % 2, torch.cuda.current_stream(self.gpu.dev)
        ev = self.ev
        if self.started[b]:
            self.up.wait_event(ev["comp"][b])
        with torch.cuda.stream(self.up):
            self.dev_in[b].copy_(self.host_in, non_blocking=True)
            ev["up"][b].record(self.up)
        comp.wait_event(ev["up"][b])
        if self.started[b]:
            comp.wait_event(ev["down"][b])
        self.graphs[b].replay()
        ev["comp"][b].record(comp)
        self.down.wait_event(ev["comp"][b])
        with torch.cuda.stream(self.down):
            self.host_out[b].copy_(self.dev_out[b], non_blocking=True)
            ev["down"][b].record(self.down)
        self.started[b] = True

    def timed(self, steps, warmup):
        torch, gpu = self.gpu.torch, self.gpu
        for c in range(warmup):
            self.chunk(c)
        torch.cuda.synchronize()
        gpu.barrier()
        comp = torch.cuda.current_stream(gpu.dev)
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(comp)
        self.up.wait_event(s)  # no upload of the timed chunks starts before the clock does
        for c in range(warmup, warmup + steps):
            self.chunk(c)
        for b in range(2):  # the last results are back on the host
            comp.wait_event(self.ev["down"][b])
        e.record(comp)
        torch.cuda.synchronize()
        gpu.barrier()
        return s.elapsed_time(e) / 1e3


def s8_peak_tops():
    """Measured dense int8 throughput of the warp-level mma.sync s8 path (libmoeq_peaks)."""
    import ctypes

    lib = ctypes.CDLL(os.path.join(ROOT, "quantized_mixture_experts_token_b300", "libmoeq_peaks.so"))
    lib.moe_peak_mma_s8.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double)]
    best = 0.0
    for _ in range(3):
        v = ctypes.c_double(0.0)
        if lib.moe_peak_mma_s8(20000, 4, ctypes.byref(v)) == 0:
            best = max(best, v.value)
    return best or None


def run_peaks():
    """--peaks: the tensor-path microbenchmarks of libmoeq_peaks, one JSON line.

    mma.sync s8 throughput, and the cycles one tcgen05.mma (M = 128, K = 16,
    fp16) costs its issuing thread at the N and the stage sizes the grouped
    prefill GEMMs use (8 or 16 MMAs per K = 64 stage)."""
    import ctypes

    import torch

    torch.cuda.init()
    lib = ctypes.CDLL(os.path.join(ROOT, "quantized_mixture_experts_token_b300", "libmoeq_peaks.so"))
    lib.moe_peak_umma_issue.argtypes = [ctypes.c_int] * 3 + [ctypes.POINTER(ctypes.c_double)]
    rows = []
    for n in (32, 64, 128, 256):
        for per_stage in (8, 16):
            for sync in (0, 1):
                v = ctypes.c_double(0.0)
                rc = lib.moe_peak_umma_issue(n, per_stage, sync, ctypes.byref(v))
                if rc != 0:
                    raise RuntimeError(f"moe_peak_umma_issue({n}, {per_stage}, {sync}) returned {rc}")
                rows.append(dict(n=n, mma_per_stage=per_stage, pipeline_sync=bool(sync), cycles_per_mma=round(v.value, 1),
                                 dense_cycles=round(128 * n * 16 / 4096, 1)))
    print(json.dumps(dict(metric="tensor_path_microbenchmarks", s8_mma_sync_tops=s8_peak_tops(), umma_issue=rows,
                          note="dense_cycles: the cycles an M=128 K=16 fp16 MMA takes at 4096 fp16 FMA (8192 FLOP) per SM per cycle")))


def distinct_experts(gpu, xs, Ws, layers, ws, nl):
    """Distinct experts the tokens of xs[l] select in layer l (read back once)."""
    out = []
    for l in range(nl):
        _, idx, _ = gpu.moeq.layer_forward(xs[l], Ws[l], layers[l].Wr, None, K_TOP, ws, residual=True,
                                           y=gpu.torch.empty_like(xs[l]), want_routing=True)
        out.append(len(set(idx.flatten().tolist())))
    return out


def decode_stack(gpu, layers, Ws, T, steps, warmup, seed, clocks=False):
    """T tokens through the nl-layer stack per step (x_{l+1} = x_l + moe_l(x_l)),
    one CUDA graph per step; returns timing, bytes and the roofline figures."""
    torch, moeq = gpu.torch, gpu.moeq
    nl = len(layers)
    ws = moeq.workspace(T, H, I, E, K_TOP, device=gpu.dev)
    xs = [torch.empty(T, H, device=gpu.dev) for _ in range(nl + 1)]
    import synth

    xs[0].copy_(synth.make_x(T, H, seed=seed, device=gpu.dev))

    def step():
        for l in range(nl):
            moeq.layer_forward(xs[l], Ws[l], layers[l].Wr, None, K_TOP, ws, residual=True, y=xs[l + 1])

    g = gpu.graph(step)
    clk = None
    if clocks:
        with ClockSampler(gpu.dev.index) as sampler:
            t = gpu.timed(g.replay, steps, warmup)
        clk = sampler.summary()
    else:
        t = gpu.timed(g.replay, steps, warmup)
    agg = aggregate(T * nl * steps, t, gpu.world)
    uniq = distinct_experts(gpu, xs, Ws, layers, ws, nl)
    layer_s = agg["seconds"] / (steps * nl)
    nbytes = ROUTER_BYTES + statistics.mean(uniq) * EXPERT_BYTES + 2 * T * H * 4
    ach = nbytes / layer_s / 1e9
    pk = gpu.pk
    roof = dict(bound="hbm", achieved=ach, peak=pk["hbm"], unit="GB/s", frac=ach / pk["hbm"],
                traffic=DECODE_LAYER_TRAFFIC["bytes"], traffic_source=DECODE_LAYER_TRAFFIC["source"],
                kernel="one decode layer: route_gemv_kernel + ffn_gemv_kernel (PDL-chained)",
                bytes_per_launch=nbytes, distinct_experts=statistics.mean(uniq), launch_us=layer_s * 1e6,
                frac_of_8tbs=ach / 8000.0, peak_source=f"{pk['source']} hbm_gbs (copy)")
    return dict(agg=agg, roof=roof, graph=g, xs=xs, ws=ws, clocks=clk, layer_us=layer_s * 1e6)


def prefill_chunk(gpu, pre_layer, preW, args, rank):
    """One 4,096-token chunk through the skewed layer: time, e2e and the
    per-kernel rooflines (router GEMM, gate/up GEMM, down GEMM)."""
    torch, moeq = gpu.torch, gpu.moeq
    import synth

    Tp = PREFILL_T
    wsp = moeq.workspace(Tp, H, I, E, K_TOP, device=gpu.dev)
    xp = synth.make_x(Tp, H, seed=21 + rank, device=gpu.dev)
    yp = torch.empty(Tp, H, device=gpu.dev)

    def call():
        moeq.layer_forward(xp, preW, pre_layer.Wr, pre_layer.bias, K_TOP, wsp, y=yp)

    g = gpu.graph(call)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    moeq.trace_events(ev)
    g_tr = gpu.graph(call)
    moeq.trace_events(None)
    psteps = max(3, args.steps // 2)
    t = gpu.timed(g.replay, psteps, args.warmup)
    pre = aggregate(Tp * psteps, t, gpu.world)
    for _ in range(3):
        g_tr.replay()
    torch.cuda.synchronize()
    rt_s, gu_s, dn_s = (ev[2 * i].elapsed_time(ev[2 * i + 1]) / 1e3 for i in range(3))
    P = Tp * K_TOP
    gu_flop, dn_flop, rt_flop = 2.0 * P * 2 * I * H, 2.0 * P * H * I, 2.0 * Tp * E * H
    pk = gpu.pk
    ach = gu_flop / gu_s / 1e12
    xh = torch.empty(Tp, H, pin_memory=True)
    xh.copy_(xp.cpu())
    yh = torch.empty(Tp, H, pin_memory=True)

    def e2e():
        xp.copy_(xh, non_blocking=True)
        g.replay()
        yh.copy_(yp, non_blocking=True)

    pe = aggregate(Tp * psteps, gpu.timed(e2e, psteps, args.warmup), gpu.world)

    # the same with the copies overlapped: chunk c's input goes up on one copy
    # stream while chunk c-1 computes, and its result comes back on another
    # while chunk c+1 computes (two device buffer pairs, one graph each)
    xp2, yp2 = torch.empty_like(xp), torch.empty_like(yp)

    def call2():
        moeq.layer_forward(xp2, preW, pre_layer.Wr, pre_layer.bias, K_TOP, wsp, y=yp2)

    pipe = Pipelined(gpu, [g, gpu.graph(call2)], [xp, xp2], [yp, yp2], xh, [yh, torch.empty_like(yh, pin_memory=True)])
    pp = aggregate(Tp * psteps, pipe.timed(psteps, args.warmup), gpu.world)
    tf32_peak = pk["bf16"] / 2.0  # tf32 dense rate is half the bf16 rate (nominal 1.1 vs 2.25 PFLOP/s)
    s8 = s8_peak_tops()

    s8_path = None if args.no_s8 else s8_chunk(gpu, call_args=(xp, preW, pre_layer, wsp, yp), psteps=psteps,
                                               args=args, s8=s8, gu_flop=gu_flop, dn_flop=dn_flop)
    return dict(
        value=pre["value"], unit="tokens/s", ms_per_chunk=1e3 * pre["seconds"] / psteps,
        workload="prefill: 4,096-token chunk through one 2048/512/512 top-10 2-bit layer, Zipf(1.1)-skewed router",
        dtype=("fp16 tensor-core products of the exact 2-bit levels and an fp16 hi/lo split of the int8 "
               "activations, fp32 accumulate; router 3xTF32"),
        roofline=dict(bound="tensor", achieved=ach, peak=pk["bf16"], unit="TFLOP/s", frac=ach / pk["bf16"],
                      traffic=GEMM_GU_TRAFFIC["bytes"], traffic_source=GEMM_GU_TRAFFIC["source"],
                      kernel="ffn_gemm_kernel<gate/up>", flop_per_launch=gu_flop, launch_us=gu_s * 1e6,
                      peak_source=f"{pk['source']} bf16_tflops (burst; fp16 = bf16 rate)",
                      note="useful FLOP; the exact hi/lo scheme issues two MMAs per product, so 0.5 is its ceiling",
                      s8_peak=dict(value=s8, unit="TOP/s", source="measured mma.sync m16n8k32 s8 (libmoeq_peaks)",
                                   frac=(ach / s8) if s8 else None),
                      down=dict(achieved=dn_flop / dn_s / 1e12, frac=dn_flop / dn_s / 1e12 / pk["bf16"],
                                launch_us=dn_s * 1e6, flop_per_launch=dn_flop),
                      router=dict(achieved=rt_flop / rt_s / 1e12, frac_of_tf32=rt_flop / rt_s / 1e12 / tf32_peak,
                                  launch_us=rt_s * 1e6, flop_per_launch=rt_flop, kernel="route_tc_kernel (3xTF32)",
                                  peak_source="tf32 = measured bf16 / 2")),
        e2e=dict(value=pp["value"], unit="tokens/s", h2d_bytes_per_step=Tp * H * 4, d2h_bytes_per_step=Tp * H * 4,
                 copies="overlapped with compute (two copy streams, double-buffered)",
                 sequential=dict(value=pe["value"], unit="tokens/s",
                                 note="copy in, compute, copy out one after another")),
        s8_path=s8_path)


def s8_chunk(gpu, call_args, psteps, args, s8, gu_flop, dn_flop):
    """The same chunk with both expert GEMMs on the warp-level int8 path (exact
    block products scaled in registers): the comparison point."""
    torch, moeq = gpu.torch, gpu.moeq
    xp, preW, pre_layer, wsp, yp = call_args
    Tp = xp.shape[0]

    def call_s8():
        moeq.layer_forward(xp, preW, pre_layer.Wr, pre_layer.bias, K_TOP, wsp, y=yp, mode=moeq.MODE_GEMM_S8)

    g8 = gpu.graph(call_s8)
    ev8 = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    moeq.trace_events(ev8)
    g8_tr = gpu.graph(call_s8)
    moeq.trace_events(None)
    pre8 = aggregate(Tp * psteps, gpu.timed(g8.replay, psteps, args.warmup), gpu.world)
    for _ in range(3):
        g8_tr.replay()
    torch.cuda.synchronize()
    gu8_s, dn8_s = (ev8[2 * i].elapsed_time(ev8[2 * i + 1]) / 1e3 for i in (1, 2))
    return dict(
        kernel="ffn_mma8_kernel: mma.sync m16n8k32 s8, every 32-block product an exact integer dot scaled in registers",
        value=pre8["value"], unit="tokens/s", ms_per_chunk=1e3 * pre8["seconds"] / psteps,
        gateup=dict(launch_us=gu8_s * 1e6, achieved_tops=gu_flop / gu8_s / 1e12,
                    frac_of_s8=(gu_flop / gu8_s / 1e12 / s8) if s8 else None),
        down=dict(launch_us=dn8_s * 1e6, achieved_tops=dn_flop / dn8_s / 1e12,
                  frac_of_s8=(dn_flop / dn8_s / 1e12 / s8) if s8 else None),
        s8_peak_tops=s8)


def stack_prompt(gpu, layers, Ws, args, rank):
    """Config of the whole model: a PROMPT_T-token prompt in PREFILL_T-token
    chunks through every layer of the stack (each chunk one CUDA graph of nl
    layer calls), then STACK_DECODE_STEPS single-token decode steps."""
    torch, moeq = gpu.torch, gpu.moeq
    import synth

    nl = len(layers)
    n_chunks = PROMPT_T // PREFILL_T
    wsp = moeq.workspace(PREFILL_T, H, I, E, K_TOP, device=gpu.dev)
    prompt = synth.make_x(PROMPT_T, H, seed=41 + rank, device=gpu.dev)
    buf = [torch.empty(PREFILL_T, H, device=gpu.dev) for _ in range(2)]

    def chunk_pass():
        for l in range(nl):
            moeq.layer_forward(buf[l & 1], Ws[l], layers[l].Wr, None, K_TOP, wsp, residual=True,
                               y=buf[(l + 1) & 1])

    g = gpu.graph(chunk_pass)

    def prompt_pass():
        for c in range(n_chunks):
            buf[0].copy_(prompt[c * PREFILL_T:(c + 1) * PREFILL_T])
            g.replay()

    reps = max(1, args.stack_reps)
    t = gpu.timed(prompt_pass, reps, 1)
    pre = aggregate(PROMPT_T * reps, t, gpu.world)
    del g, wsp, buf, prompt
    torch.cuda.empty_cache()
    dec = decode_stack(gpu, layers, Ws, 1, STACK_DECODE_STEPS, args.warmup, seed=51 + rank)
    return dict(
        workload=(f"{PROMPT_T}-token prompt in {n_chunks} chunks of {PREFILL_T} through {nl} layers "
                  f"(uniform routing, residual between layers), then {STACK_DECODE_STEPS} decode steps of one token"),
        prefill=dict(value=pre["value"], unit="prompt tokens/s through the stack",
                     ms_per_prompt=1e3 * pre["seconds"] / reps, reps=reps),
        decode=dict(value=dec["agg"]["value"] / nl, unit="tokens/s through the stack",
                    ms_per_token=1e3 * dec["agg"]["seconds"] / STACK_DECODE_STEPS, steps=STACK_DECODE_STEPS,
                    roofline_frac=dec["roof"]["frac"]))


def bits3_section(gpu, args, rank):
    torch, moeq = gpu.torch, gpu.moeq
    import synth

    pk = gpu.pk
    l3 = synth.make_layer(synth.FULL3, seed=0, layer=2000, device=gpu.dev)
    W3 = moeq.ExpertWeights.from_layer(l3)
    torch.cuda.synchronize()
    res = {}
    for name, T3 in (("decode", VERIFY_T), ("prefill", PREFILL3_T)):
        ws3 = moeq.workspace(T3, H, I, E, K_TOP, bits=3, device=gpu.dev)
        x3 = synth.make_x(T3, H, seed=31 + rank, device=gpu.dev)
        y3 = torch.empty(T3, H, device=gpu.dev)
        _, idx3, _ = moeq.layer_forward(x3, W3, l3.Wr, None, K_TOP, ws3, y=y3, want_routing=True)
        g3 = gpu.graph(lambda: moeq.layer_forward(x3, W3, l3.Wr, None, K_TOP, ws3, y=y3))
        n3 = max(3, args.steps // 2)
        t3 = aggregate(T3 * n3, gpu.timed(g3.replay, n3, args.warmup), gpu.world)
        sec = t3["seconds"] / n3
        if name == "decode":
            uniq = len(set(idx3.flatten().tolist()))
            nbytes = ROUTER_BYTES + uniq * EXPERT_BYTES3 + 2 * T3 * H * 4
            ach = nbytes / sec / 1e9
            roof = dict(bound="hbm", achieved=ach, peak=pk["hbm"], unit="GB/s", frac=ach / pk["hbm"], traffic=None,
                        kernel="whole layer call (router + expert kernels)", bytes_per_launch=nbytes,
                        distinct_experts=uniq, peak_source=f"{pk['source']} hbm_gbs (copy)")
        else:
            flop = 2.0 * T3 * K_TOP * 3 * H * I
            ach = flop / sec / 1e12
            roof = dict(bound="tensor", achieved=ach, peak=pk["bf16"], unit="TFLOP/s", frac=ach / pk["bf16"],
                        traffic=None, kernel="whole layer call (router, permutation, both GEMMs)",
                        flop_per_launch=flop, peak_source=f"{pk['source']} bf16_tflops (burst)")
        res[name] = dict(T=T3, value=t3["value"], unit="tokens/s", ms_per_call=1e3 * sec, roofline=roof)
        del ws3, x3, y3, g3
    return dict(workload="3-bit block-32 weights, one 2048/512/512 top-10 layer, uniform routing",
                dtype="3-bit x int8 block dots (decode); fp16 tensor-core products of exact hi/lo operands (prefill)",
                **res)


def mode_sweep(gpu, layers, Ws, args):
    """Whole-layer time per call in GEMV and in grouped-GEMM mode for small T,
    each replay running all resident layers so the experts come from HBM."""
    torch, moeq = gpu.torch, gpu.moeq
    import synth

    nl = len(layers)
    rows = []
    for Ts in SWEEP_T:
        wss = moeq.workspace(Ts, H, I, E, K_TOP, device=gpu.dev)
        xsw = synth.make_x(Ts, H, seed=61 + Ts, device=gpu.dev)
        ysw = torch.empty(Ts, H, device=gpu.dev)
        row = dict(T=Ts)
        for mname, mode in (("gemv", moeq.MODE_GEMV), ("gemm", moeq.MODE_GEMM)):
            def stack(mode=mode):
                for l in range(nl):
                    moeq.layer_forward(xsw, Ws[l], layers[l].Wr, None, K_TOP, wss, y=ysw, mode=mode)

            gs = gpu.graph(stack)
            nrep = 5
            row[mname + "_us_per_layer"] = 1e6 * gpu.timed(gs.replay, nrep, args.warmup) / (nrep * nl)
            del gs
        row["faster"] = "gemv" if row["gemv_us_per_layer"] <= row["gemm_us_per_layer"] else "gemm"
        rows.append(row)
        del wss, xsw, ysw
    return rows


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)

    import __graft_entry__

    __graft_entry__.build()
    import synth

    gpu = Gpu(world, local)
    moeq = gpu.moeq
    shape = synth.FULL
    nl = args.layers

    # ---- resident weights: nl decode layers + one skewed prefill layer
    layers = [synth.make_layer(shape, seed=0, layer=l, device=gpu.dev) for l in range(nl)]
    Ws = [moeq.ExpertWeights.from_layer(l) for l in layers]
    pre_layer = synth.make_layer(shape, seed=0, layer=1000, device=gpu.dev, skew=True)
    preW = moeq.ExpertWeights.from_layer(pre_layer)
    torch.cuda.synchronize()

    # ---- headline: B=1 decode through the stack
    dec = decode_stack(gpu, layers, Ws, DECODE_T, args.steps, args.warmup, seed=11 + rank, clocks=True)
    T = DECODE_T
    x_host = torch.empty(T, H, pin_memory=True)
    x_host.copy_(dec["xs"][0].cpu())
    y_host = torch.empty(T, H, pin_memory=True)

    def e2e_step():  # pinned host token in, result out, every step
        dec["xs"][0].copy_(x_host, non_blocking=True)
        dec["graph"].replay()
        y_host.copy_(dec["xs"][nl], non_blocking=True)

    dec_e2e = aggregate(T * nl * args.steps, gpu.timed(e2e_step, args.steps, args.warmup), world)

    # ---- 8 tokens per decode call through the stack
    d8 = decode_stack(gpu, layers, Ws, DECODE_T8, args.steps, args.warmup, seed=13 + rank)
    decode_t8 = dict(T=DECODE_T8, value=d8["agg"]["value"], unit="layer-tokens/s",
                     us_per_layer=d8["layer_us"], roofline=d8["roof"])
    del d8

    prefill = None if args.no_prefill else prefill_chunk(gpu, pre_layer, preW, args, rank)
    stack = None if args.no_stack else stack_prompt(gpu, layers, Ws, args, rank)
    bits3 = None if args.no_3bit else bits3_section(gpu, args, rank)
    sweep = None if args.no_sweep else mode_sweep(gpu, layers, Ws, args)

    status = moeq.device_status()
    if status:
        raise SystemExit(f"device status 0x{status:x}")

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        lnp = layers[0].numpy()
        n_tok = args.ref_tokens
        r, threads, dt = oracle_decode_rate(lnp, n_tok)
        cpu = dict(value=r, unit="tokens/s", cores=threads, kind="oracle",
                   sample=f"{n_tok} independent B=1 decode tokens through one layer ({dt:.1f} s wall)")

    launches_per_step = 2 * nl  # router kernel + expert kernel per layer
    line = dict(
        metric=METRIC, value=dec["agg"]["value"], unit="tokens/s", n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=1e3 * dec["agg"]["seconds"] / args.steps, higher_is_better=True,
        scaling="weak", vs_baseline=None, dtype="int8 x 2-bit integer block dots, fp32 scales", data="synthetic",
        config=dict(workload=(f"decode: B=1 token through {nl} resident MoE layers (H=2048, E=512, I=512, top-10, "
                              "2-bit block-32 weights, residual between layers); value = per-layer tokens/s"),
                    T=DECODE_T, layers=nl, stack_tokens_per_s=dec["agg"]["value"] / nl,
                    l2="inputs larger than L2: every step reads the selected experts of 48 distinct layers",
                    parallelism=f"replicas x{world}"),
        roofline=dec["roof"], cpu_baseline=cpu,
        e2e=dict(value=dec_e2e["value"], unit="tokens/s", h2d_bytes_per_step=T * H * 4, d2h_bytes_per_step=T * H * 4),
        gpu_launches=launches_per_step * args.steps, clocks=dec["clocks"], decode_t8=decode_t8, prefill=prefill,
        stack=stack, bits3=bits3, mode_sweep=sweep)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--layers", type=int, default=N_LAYERS)
    ap.add_argument("--ref-tokens", type=int, default=32)
    ap.add_argument("--stack-reps", type=int, default=2)
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-s8", action="store_true", help="skip the int8 comparison leg of the prefill chunk")
    ap.add_argument("--no-stack", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-3bit", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--peaks", action="store_true", help="only run the tensor-path microbenchmarks")
    args = ap.parse_args(argv)
    if args.peaks:
        run_peaks()
        return
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Throughput of the routed expert-FFN layer on B300.

Headline workload (one JSON line on stdout, rank 0):
  decode -- one token (B=1) through a stack of 48 resident MoE layers
            (H=2048, E=512, I=512, top-10, 2-bit block-32 weights, residual
            add between layers); `value` is per-layer tokens/s, i.e. tokens
            through one layer per second, measured over the whole stack so
            every step reads 48 distinct layers' experts (~673 MB > L2).
  prefill -- a 4,096-token chunk through one such layer whose router bias is
            Zipf-skewed (some experts get no token), reported in the "prefill"
            object (inputs 0.57 GB > L2).
Both are replayed from CUDA graphs of the library's C-ABI calls.  The
expert kernels' device time comes from CUDA events the library records
around them (moe_trace_events); roofline fractions use MEASURED_PEAKS.json.

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
PREFILL_T = 4096
EXPERT_BYTES = 3 * I * (H // 32) * (8 + 2)  # 2-bit codes + fp16 scales of gate, up, down = 983,040
EXPERT_BYTES3 = 3 * I * (H // 32) * (12 + 2)  # 3-bit: 1,376,256
VERIFY_T = 64  # 3-bit decode: a multi-token verify window
PREFILL3_T = 16384  # 3-bit prefill chunk, uniform routing
SWEEP_T = (8, 16, 32, 64, 128, 256, 512, 1024)  # token counts of the GEMV / grouped-GEMM crossover sweep
# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) that ncu
# measured for the current kernel versions on this workload (cold caches): the
# decode expert kernel (10 experts, T=1) and the prefill gate/up GEMM
GEMV_TRAFFIC_BYTES = 9.92e6
GEMM_GU_TRAFFIC_BYTES = 690.0e6 + 19.6e6
# library kernels per prefill chunk: router SGEMM, top-k, 3 permutation kernels,
# plan, y init, x quantisation, 2 operand images, 2 GEMMs
PREFILL_LAUNCHES = 12


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


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__

    __graft_entry__.build()
    import quantized_mixture_experts_token_b300 as moeq
    import synth

    pk = peaks()
    shape = synth.FULL
    nl = args.layers

    def barrier():
        if world > 1:
            import torch.distributed as dist

            dist.barrier()

    # ---- resident weights: nl decode layers + one skewed prefill layer
    layers = [synth.make_layer(shape, seed=0, layer=l, device=dev) for l in range(nl)]
    Ws = [moeq.ExpertWeights.from_layer(l) for l in layers]
    pre_layer = synth.make_layer(shape, seed=0, layer=1000, device=dev, skew=True)
    preW = moeq.ExpertWeights.from_layer(pre_layer)
    torch.cuda.synchronize()

    # ---- decode: one token through the stack, residual chain x_{l+1} = x_l + moe_l(x_l)
    T = DECODE_T
    ws = moeq.workspace(T, H, I, E, K_TOP, device=dev)
    xs = [torch.empty(T, H, device=dev) for _ in range(nl + 1)]
    xs[0].copy_(synth.make_x(T, H, seed=11 + rank, device=dev))

    def decode_pass():
        for l in range(nl):
            moeq.layer_forward(xs[l], Ws[l], layers[l].Wr, None, K_TOP, ws, residual=True, y=xs[l + 1])

    decode_pass()
    torch.cuda.synchronize()
    g_dec = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_dec):
        decode_pass()
    # a second graph whose expert-kernel launches are bracketed by events
    ev_dec = [torch.cuda.Event(enable_timing=True) for _ in range(2 * nl)]
    moeq.trace_events(ev_dec)
    g_dec_tr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_dec_tr):
        decode_pass()
    moeq.trace_events(None)

    def timed(fn, steps, warmup):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        barrier()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        barrier()
        return s.elapsed_time(e) / 1e3

    with ClockSampler(local) as clk:
        t_dec = timed(g_dec.replay, args.steps, args.warmup)
    clocks = clk.summary()
    dec = aggregate(T * nl * args.steps, t_dec, world)

    # expert-kernel time per launch (traced graph, replayed after warm-up)
    for _ in range(3):
        g_dec_tr.replay()
    torch.cuda.synchronize()
    k_ms = [ev_dec[2 * l].elapsed_time(ev_dec[2 * l + 1]) for l in range(nl)]
    gemv_s = statistics.mean(k_ms) / 1e3
    # algorithmic bytes of one decode expert launch: the selected experts' weights once
    uniq = []
    for l in range(nl):
        _, idx, _ = moeq.layer_forward(xs[l], Ws[l], layers[l].Wr, None, K_TOP, ws, residual=True,
                                       y=torch.empty_like(xs[l]), want_routing=True)
        uniq.append(len(set(idx.flatten().tolist())))
    dec_bytes = statistics.mean(uniq) * EXPERT_BYTES + 2 * T * H * 4
    achieved = dec_bytes / gemv_s / 1e9
    roof_dec = dict(bound="hbm", achieved=achieved, peak=pk["hbm"], unit="GB/s", frac=achieved / pk["hbm"],
                    traffic=GEMV_TRAFFIC_BYTES, kernel="ffn_gemv_kernel<2>", bytes_per_launch=dec_bytes,
                    launch_us=gemv_s * 1e6, peak_source=f"{pk['source']} hbm_gbs (copy)")

    # decode end to end: pinned host token in, result out, every step
    x_host = torch.empty(T, H, pin_memory=True)
    x_host.copy_(xs[0].cpu())
    y_host = torch.empty(T, H, pin_memory=True)

    def e2e_step():
        xs[0].copy_(x_host, non_blocking=True)
        g_dec.replay()
        y_host.copy_(xs[nl], non_blocking=True)

    t_e2e = timed(e2e_step, args.steps, args.warmup)
    dec_e2e = aggregate(T * nl * args.steps, t_e2e, world)

    # ---- prefill: a 4,096-token chunk through the skewed layer
    out = {}
    if not args.no_prefill:
        Tp = PREFILL_T
        wsp = moeq.workspace(Tp, H, I, E, K_TOP, device=dev)
        xp = synth.make_x(Tp, H, seed=21 + rank, device=dev)
        yp = torch.empty(Tp, H, device=dev)

        def prefill_call():
            moeq.layer_forward(xp, preW, pre_layer.Wr, pre_layer.bias, K_TOP, wsp, y=yp)

        prefill_call()
        torch.cuda.synchronize()
        g_pre = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pre):
            prefill_call()
        ev_pre = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        moeq.trace_events(ev_pre)
        g_pre_tr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pre_tr):
            prefill_call()
        moeq.trace_events(None)
        psteps = max(3, args.steps // 2)
        t_pre = timed(g_pre.replay, psteps, args.warmup)
        pre = aggregate(Tp * psteps, t_pre, world)
        for _ in range(3):
            g_pre_tr.replay()
        torch.cuda.synchronize()
        gu_s = ev_pre[0].elapsed_time(ev_pre[1]) / 1e3
        dn_s = ev_pre[2].elapsed_time(ev_pre[3]) / 1e3
        P = Tp * K_TOP
        gu_flop = 2.0 * P * 2 * I * H
        dn_flop = 2.0 * P * H * I
        ach = gu_flop / gu_s / 1e12
        xp_host = torch.empty(Tp, H, pin_memory=True)
        xp_host.copy_(xp.cpu())
        yp_host = torch.empty(Tp, H, pin_memory=True)

        def pre_e2e():
            xp.copy_(xp_host, non_blocking=True)
            g_pre.replay()
            yp_host.copy_(yp, non_blocking=True)

        t_pe = timed(pre_e2e, psteps, args.warmup)
        pre_e2e_v = aggregate(Tp * psteps, t_pe, world)
        out = dict(
            value=pre["value"], unit="tokens/s", ms_per_chunk=1e3 * pre["seconds"] / psteps,
            workload="prefill: 4,096-token chunk through one 2048/512/512 top-10 2-bit layer, Zipf(1.1)-skewed router",
            dtype="fp16 tensor-core products of the exact 2-bit levels and an fp16 hi/lo split of the int8 activations, fp32 accumulate",
            roofline=dict(bound="tensor", achieved=ach, peak=pk["bf16"], unit="TFLOP/s", frac=ach / pk["bf16"],
                          traffic=GEMM_GU_TRAFFIC_BYTES, kernel="ffn_gemm_kernel<gate/up>", flop_per_launch=gu_flop,
                          launch_us=gu_s * 1e6, peak_source=f"{pk['source']} bf16_tflops (burst; fp16 = bf16 rate)",
                          down=dict(achieved=dn_flop / dn_s / 1e12, launch_us=dn_s * 1e6, flop_per_launch=dn_flop)),
            e2e=dict(value=pre_e2e_v["value"], unit="tokens/s", h2d_bytes_per_step=Tp * H * 4,
                     d2h_bytes_per_step=Tp * H * 4),
            gpu_launches_per_chunk=PREFILL_LAUNCHES)

    # ---- 3-bit weights: a 64-token verify window (decode path) and a 16,384-token
    # prefill chunk, one layer with uniform routing (no bias)
    bits3 = None
    if not args.no_3bit:
        l3 = synth.make_layer(synth.FULL3, seed=0, layer=2000, device=dev)
        W3 = moeq.ExpertWeights.from_layer(l3)
        torch.cuda.synchronize()
        res3 = {}
        for name, T3 in (("decode", VERIFY_T), ("prefill", PREFILL3_T)):
            ws3 = moeq.workspace(T3, H, I, E, K_TOP, bits=3, device=dev)
            x3 = synth.make_x(T3, H, seed=31 + rank, device=dev)
            y3 = torch.empty(T3, H, device=dev)
            _, idx3, _ = moeq.layer_forward(x3, W3, l3.Wr, None, K_TOP, ws3, y=y3, want_routing=True)
            torch.cuda.synchronize()
            g3 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g3):
                moeq.layer_forward(x3, W3, l3.Wr, None, K_TOP, ws3, y=y3)
            n3 = max(3, args.steps // 2)
            t3 = aggregate(T3 * n3, timed(g3.replay, n3, args.warmup), world)
            sec = t3["seconds"] / n3
            if name == "decode":
                uniq = len(set(idx3.flatten().tolist()))
                nbytes = E * H * 4 + uniq * EXPERT_BYTES3 + 2 * T3 * H * 4
                ach = nbytes / sec / 1e9
                roof = dict(bound="hbm", achieved=ach, peak=pk["hbm"], unit="GB/s", frac=ach / pk["hbm"],
                            traffic=None, kernel="whole layer call (router + expert kernels)",
                            bytes_per_launch=nbytes, distinct_experts=uniq,
                            peak_source=f"{pk['source']} hbm_gbs (copy)")
            else:
                flop = 2.0 * T3 * K_TOP * 3 * H * I
                ach = flop / sec / 1e12
                roof = dict(bound="tensor", achieved=ach, peak=pk["bf16"], unit="TFLOP/s", frac=ach / pk["bf16"],
                            traffic=None, kernel="whole layer call (router, permutation, both GEMMs)",
                            flop_per_launch=flop, peak_source=f"{pk['source']} bf16_tflops (burst)")
            res3[name] = dict(T=T3, value=t3["value"], unit="tokens/s", ms_per_call=1e3 * sec, roofline=roof)
            del ws3, x3, y3, g3
        bits3 = dict(workload="3-bit block-32 weights, one 2048/512/512 top-10 layer, uniform routing",
                     dtype="3-bit x int8 block dots (decode); fp16 tensor-core products of exact hi/lo operands (prefill)",
                     **res3)
        del l3, W3

    # ---- expert-path crossover: whole-layer time per call in GEMV and in grouped-GEMM
    # mode for small T, each replay running all nl resident layers so the selected
    # experts come from HBM, not L2
    sweep = None
    if not args.no_sweep:
        sweep = []
        for Ts in SWEEP_T:
            wss = moeq.workspace(Ts, H, I, E, K_TOP, device=dev)
            xsw = synth.make_x(Ts, H, seed=61 + Ts, device=dev)
            ysw = torch.empty(Ts, H, device=dev)
            row = dict(T=Ts)
            for mname, mode in (("gemv", moeq.MODE_GEMV), ("gemm", moeq.MODE_GEMM)):
                def stack(mode=mode):
                    for l in range(nl):
                        moeq.layer_forward(xsw, Ws[l], layers[l].Wr, None, K_TOP, wss, y=ysw, mode=mode)

                stack()
                torch.cuda.synchronize()
                gs = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gs):
                    stack()
                nrep = 5
                row[mname + "_us_per_layer"] = 1e6 * timed(gs.replay, nrep, args.warmup) / (nrep * nl)
                del gs
            row["faster"] = "gemv" if row["gemv_us_per_layer"] <= row["gemm_us_per_layer"] else "gemm"
            sweep.append(row)
            del wss, xsw, ysw

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

    launches_per_step = 2 * nl  # fused routing kernel + expert GEMV per layer
    line = dict(
        metric=METRIC, value=dec["value"], unit="tokens/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
        ms_per_step=1e3 * dec["seconds"] / args.steps, higher_is_better=True, scaling="weak", vs_baseline=None,
        dtype="int8 x 2-bit integer block dots, fp32 scales", data="synthetic",
        config=dict(workload=(f"decode: B=1 token through {nl} resident MoE layers (H=2048, E=512, I=512, top-10, "
                              "2-bit block-32 weights, residual between layers); value = per-layer tokens/s"),
                    T=DECODE_T, layers=nl, stack_tokens_per_s=dec["value"] / nl,
                    l2="inputs larger than L2: every step reads the selected experts of 48 distinct layers",
                    parallelism=f"replicas x{world}"),
        roofline=roof_dec, cpu_baseline=cpu,
        e2e=dict(value=dec_e2e["value"], unit="tokens/s", h2d_bytes_per_step=T * H * 4, d2h_bytes_per_step=T * H * 4),
        gpu_launches=launches_per_step * args.steps, clocks=clocks, prefill=out or None, bits3=bits3,
        mode_sweep=sweep)
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
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-3bit", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

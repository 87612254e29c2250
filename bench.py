"""Benchmark: one dropless-MoE layer fwd+bwd step (route, permute, MXFP8
quantize, grouped GEMMs with fused SwiGLU, combine, and the backward of each)
on the DeepSeek-V3-shaped workload: T = 24576 tokens (6 x 4096), d = 7168,
E = 256 routed experts, top-8 sigmoid routing with normalised weights,
f = 2048, R = T*k = 196,608 routed rows, bf16 activations, MXFP8 operands.

Prints ONE JSON line (rank 0).  `value` = fwd+bwd grouped-GEMM TFLOPS
(18*R*d*f algorithmic FLOPs per step / device time per step), whole job.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload deepseek-v3|mixtral|tiny] [--no-cpu-baseline]

--impl reference times the CPU oracle (plain fp64 numpy) on a bounded sample
of the same workload: the only other place this file runs oracle code.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOADS = {
    # name: T, d, E, k, f, score, normalize, zipf
    "deepseek-v3": dict(T=24576, d=7168, E=256, k=8, f=2048, score="sigmoid", normalize=True, zipf=None,
                        desc="DeepSeek-V3-shaped routed-expert layer fwd+bwd: T=24576 (6x4096), d=7168, E=256, "
                             "top-8 sigmoid normalised, f=2048"),
    "deepseek-v3-small": dict(T=1536, d=7168, E=16, k=8, f=2048, score="sigmoid", normalize=True, zipf=None,
                              desc="DeepSeek-V3 expert shapes with 16 experts and 1536 tokens (same 768 rows per "
                                   "expert; profiling case): d=7168, top-8 sigmoid, f=2048"),
    "deepseek-v3-zipf": dict(T=24576, d=7168, E=256, k=8, f=2048, score="sigmoid", normalize=True, zipf=1.2,
                             desc="DeepSeek-V3-shaped layer fwd+bwd with Zipf(1.2)-skewed routing (logit bias "
                                  "-1.2 ln rank_e, rank a seeded permutation): T=24576, d=7168, E=256, top-8 "
                                  "sigmoid normalised, f=2048"),
    "mixtral": dict(T=8192, d=4096, E=8, k=2, f=14336, score="softmax", normalize=True, zipf=None,
                    desc="Mixtral-shaped layer fwd+bwd: T=8192, d=4096, E=8, top-2 softmax, f=14336"),
    "tiny": dict(T=256, d=512, E=8, k=2, f=256, score="softmax", normalize=True, zipf=None,
                 desc="tiny layer fwd+bwd: T=256, d=512, E=8, top-2, f=256"),
}
METRIC = "MoE layer fwd+bwd TFLOPS (MXFP8 grouped GEMM) and % of dense peak, 1 GB300"
KERNELS_PER_STEP = 18       # libmoe kernel launches in one fwd+bwd step (see layer.MoELayer)
WGRAD_SPLIT_KERNELS = 2     # a second launch per weight gradient when they are split by group size
ROUTER_KERNELS = 6          # with the router: 3 bf16 GEMMs, 3 transposes (the dx combine takes the addend)
GEMMS_PER_STEP = 6


def _gemm_traffic():
    """DRAM bytes per grouped-GEMM launch from the committed ncu summary
    (profiles/gemm_traffic.json), only if the GEMM sources are unchanged
    since those counters were taken; else None."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_traffic.json")) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for fn in ["common.cuh", "gemm_common.cuh", "gemm.cu", "gemm2sm.cu"]:
            with open(os.path.join(ROOT, "grouped_gemm_top_gb300", "csrc", fn), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != rec["kernel_source_hash"]:
            return None
        return rec["gemm_launches"]
    except Exception:
        return None


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "sm_max_mhz": 2070.0}, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 200 ms in a thread."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.idx)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        pw = [float(r[3]) for r in self.rows if r[3].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows), "power_w_max": max(pw) if pw else None}


# --------------------------------------------------------------------- GPU --

def run_gpu(args, rank, world, local_rank):
    import torch

    from grouped_gemm_top_gb300 import build as _b
    if not os.path.exists(_b.LIB):
        _b.build()
    from grouped_gemm_top_gb300 import synth
    from grouped_gemm_top_gb300.layer import MoELayer

    torch.cuda.set_device(local_rank)
    dev = f"cuda:{local_rank}"
    w = WORKLOADS[args.workload]
    T, d, E, k, f = w["T"], w["d"], w["E"], w["k"], w["f"]
    S = args.shared_experts
    L = MoELayer(T, d, E, k, f, w["score"], w["normalize"], device=dev, router=args.router, n_shared=S,
                 wgrad224_rows=args.wgrad224_rows)
    if args.router:
        L.set_router_weights(synth.make_normal_bf16((d, E), 5, dev, std=0.02))
    inp = synth.make_layer_inputs(T, d, E, f, dev, zipf_s=w["zipf"], seed_offset=rank, n_shared=S)
    L.set_weights(inp["W1"], inp["W2"])
    del inp["W1"], inp["W2"]
    L.logits.copy_(inp["logits"])
    L.x.copy_(inp["x"])
    L.dout.copy_(inp["dout"])
    torch.cuda.synchronize()
    flops = L.flops_per_step()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # per-GEMM events: the GEMM launches of a step, in issue order
    gemm_names = ["up_fwd_swiglu", "down_fwd", "down_dgrad", "down_wgrad", "up_dgrad", "up_wgrad"]
    gemm_flops = [4 * L.R * d * f, 2 * L.R * d * f, 2 * L.R * d * f, 2 * L.R * d * f, 4 * L.R * d * f,
                  4 * L.R * d * f]
    for _ in range(args.warmup):
        L.step_()
    torch.cuda.synchronize()
    L.check_err()

    # ---- timed region: K eager steps, events around every GEMM launch
    ev_pairs = []
    L.gemm_events = ev_pairs
    L.mem_events = {}
    rev_pairs = []
    if args.router:
        L.router_events = rev_pairs
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        barrier()
        torch.cuda.synchronize()
        t_start.record(stream)
        for _ in range(args.steps):
            L.step_()
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier()
    L.gemm_events = None
    L.router_events = None
    mem_events, L.mem_events = L.mem_events, None
    L.check_err()
    mem_ms = {n: sum(s_.elapsed_time(e_) for s_, e_ in evs) / args.steps for n, evs in mem_events.items()}
    Rp = int(L.gofs[-1].item())
    elapsed_ms = t_start.elapsed_time(t_end)
    gemm_ms = [0.0] * GEMMS_PER_STEP
    for i, (s, e) in enumerate(ev_pairs):
        gemm_ms[i % GEMMS_PER_STEP] += s.elapsed_time(e)
    gemm_ms = [x / args.steps for x in gemm_ms]

    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    ms_per_step = elapsed_ms / args.steps

    # ---- CUDA-graph replay of the same step (the whole step in one graph)
    L.capture()
    for _ in range(2):
        L.replay()
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        L.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    L.check_err()
    graph_ms = max_over_ranks(g0.elapsed_time(g1), world, dev) / args.steps

    # ---- end to end through the public API from pinned host buffers
    h_x = inp["x"].cpu().pin_memory()
    h_l = inp["logits"].cpu().pin_memory()
    h_d = inp["dout"].cpu().pin_memory()
    h_out = torch.empty((T, d), dtype=torch.bfloat16).pin_memory()
    h_dx = torch.empty((T, d), dtype=torch.bfloat16).pin_memory()
    h_dl = torch.empty((T, E), dtype=torch.float32).pin_memory()
    # steps through MoELayer.run_pipelined: every step copies its inputs in
    # and its outputs out; step i+1's input copy and step i-1's output copy
    # overlap step i's kernels (three sets of device inputs and outputs)
    batch = (h_x, h_l, h_d, h_out, h_dx, h_dl)
    L.run_pipelined([batch] * 3)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk_e2e:
        barrier()
        e0.record(stream)
        L.run_pipelined([batch] * args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    h2d = h_x.numel() * 2 + h_l.numel() * 4 + h_d.numel() * 2
    d2h = h_out.numel() * 2 + h_dx.numel() * 2 + h_dl.numel() * 4

    # the host link alone (same pinned buffers, no kernels): end to end is
    # bounded by max(device step, copy time) when the copies overlap
    def link_ms(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(reps):
            fn()
        c1.record(stream)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1) / reps

    h2d_ms = link_ms(lambda: (L.x.copy_(h_x, non_blocking=True), L.logits.copy_(h_l, non_blocking=True),
                              L.dout.copy_(h_d, non_blocking=True)))
    d2h_ms = link_ms(lambda: (h_out.copy_(L.out, non_blocking=True), h_dx.copy_(L.dx, non_blocking=True),
                              h_dl.copy_(L.dlogits, non_blocking=True)))

    peaks, psrc = _peaks()
    # the GEMM launches are timed one by one (2.5-6 ms each): the burst peak;
    # the sustained one (a seconds-long loop under the power cap) beside it
    mx_peak = 2.0 * peaks["bf16_tflops"]               # nominal fp8/bf16 dense ratio 4.5/2.25
    mx_peak_sus = 2.0 * peaks["bf16_tflops_sustained"]
    write_ceiling = hbm_write_ceiling(dev)
    traffic = _gemm_traffic() if args.workload == "deepseek-v3" and not S else None
    # algorithmic bytes of the six GEMMs: fp8 operands (+1/32 scales) once,
    # bf16 outputs (and the SwiGLU-bwd input a_pre) once, h as its MXFP8
    # codes on both axes
    R, q, Gw = L.R, 1 + 1 / 32, L.G          # rows and weight groups include the shared experts
    algo_bytes = (R * d * q + Gw * d * 2 * f * q + R * 2 * f * 2 + 2 * R * f * q        # up fwd + SwiGLU + MXFP8(h)
                  + R * f * q + Gw * f * d * q + R * d * 2                               # down fwd
                  + R * d * q + Gw * f * d * q + R * f * 4                               # down dgrad (fp32 dH)
                  + R * f * q + R * d * q + Gw * f * d * 2                               # dW2
                  + R * 2 * f * q + Gw * d * 2 * f * q + R * d * 2                       # up dgrad
                  + R * d * q + R * 2 * f * q + Gw * d * 2 * f * 2)                      # dW1
    sum_gemm_ms = sum(gemm_ms)
    achieved = sum(gemm_flops) / (sum_gemm_ms * 1e-3) / 1e12
    per_launch = {n: {"ms": round(t, 4), "tflops": round(fl / (t * 1e-3) / 1e12, 1)}
                  for n, t, fl in zip(gemm_names, gemm_ms, gemm_flops)}
    value = job_tflops(flops, world, ms_per_step)
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp8(e4m3,e8m0) x mxfp8 -> fp32 acc -> bf16",
        "data": "synthetic (seeded N(0,1) activations/logits, N(0,0.02^2) weights, random-init)",
        "config": {"workload": w["desc"], "global_batch": T * world, "seq_len": 4096,
                   "parallelism": f"replicas x{world} (no collectives)", "routed_rows": L.R,
                   "row_capacity": L.row_cap,
                   "l2": "no flush: inputs and weights (~45 GB) far exceed the 129 MB L2"},
        "tokens_per_s": round(world * T / (ms_per_step * 1e-3), 1),
        "frac_of_dense_mxfp8_peak": round(value / mx_peak, 4),
        "frac_of_dense_mxfp8_peak_sustained": round(value / mx_peak_sus, 4),
        "graph_ms_per_step": round(graph_ms, 4),
        "gemm_per_launch": per_launch,
        "roofline": {"bound": "tensor", "kernel": "k_grouped_gemm (all 6 launches of a step)",
                     "achieved": round(achieved, 1), "peak": round(mx_peak, 1), "unit": "TFLOP/s",
                     "frac": round(achieved / mx_peak, 4),
                     "peak_source": f"2 x {psrc} bf16 burst ({peaks['bf16_tflops']} TF/s), "
                                    "nominal MXFP8/bf16 dense ratio 4.5/2.25 (launches timed one by one)",
                     "frac_of_sustained": round(achieved / mx_peak_sus, 4),
                     "sustained_peak": round(mx_peak_sus, 1),
                     "sustained_note": f"2 x {psrc} bf16 sustained ({peaks['bf16_tflops_sustained']} TF/s, a "
                                       f"seconds-long loop at {peaks.get('clocks_under_load', {}).get('sm_mhz_median')}"
                                       f" MHz median SM clock); this run's median SM clock is in 'clocks'",
                     "traffic": (None if traffic is None else
                                 round(sum(t["dram_read"] + t["dram_write"] for t in traffic) / len(traffic))),
                     "traffic_unit": "bytes per launch (DRAM read+write, ncu, mean of the step's 6 launches)",
                     "algorithmic_bytes_per_launch": round(algo_bytes / GEMMS_PER_STEP)},
        "e2e": {"value": round(job_tflops(flops, world, e2e_ms), 2), "unit": "TFLOPS",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "h2d_gbs": round(h2d / (h2d_ms * 1e-3) / 1e9, 1), "d2h_gbs": round(d2h / (d2h_ms * 1e-3) / 1e9, 1),
                "clocks": clk_e2e.summary()},
        "roofline_memory": memory_roofline(L, mem_ms, Rp, peaks, psrc, write_ceiling),
        "gpu_launches": (KERNELS_PER_STEP + (ROUTER_KERNELS if args.router else 0) + (2 if S else 0) +
                         (WGRAD_SPLIT_KERNELS if L.wgrad_split else 0)) * args.steps,
        "clocks": clk.summary(),
    }
    if args.router:
        rnames = ["logits = x W_r", "dx_r = dlogits W_r^T", "dW_r = x^T dlogits"]
        rms = [0.0] * 3
        for i, (s_, e_) in enumerate(rev_pairs):
            rms[i % 3] += s_.elapsed_time(e_)
        rms = [x / args.steps for x in rms]
        rflops = 2.0 * T * d * E
        bf_peak = peaks["bf16_tflops_sustained"]
        result["router"] = {
            "included_in_step": True,
            "gemm_per_launch": {n: {"ms": round(t, 4), "tflops": round(rflops / (t * 1e-3) / 1e12, 1)}
                                for n, t in zip(rnames, rms)},
            "roofline": {"bound": "tensor (bf16, kind::f16)", "achieved": round(3 * rflops / (sum(rms) * 1e-3) / 1e12, 1),
                         "peak": bf_peak, "unit": "TFLOP/s",
                         "frac": round(3 * rflops / (sum(rms) * 1e-3) / 1e12 / bf_peak, 4),
                         "peak_source": f"{psrc} bf16 sustained"},
            "flops_per_step": 3 * rflops,
        }
        result["config"]["router"] = "logits = x W_r (bf16 [d, E]) inside the step, with its backward"
    if S:
        result["config"]["shared_experts"] = (f"{S} shared expert(s) of the routed experts' shape, every token, "
                                              f"weight 1: {L.G} expert groups, {L.kk} rows per token")
    return result, L


def hbm_write_ceiling(device, nbytes=4 << 30, reps=5):
    """The GPU's write-only bandwidth with the library's own write stream
    (moe_hbm_fill: 16-byte vector stores, and bulk copies out of shared
    memory); the better of the two, best of `reps` after 3 warm-ups (CUDA
    events on the launching stream, 4 GB: far above L2)."""
    import torch

    from grouped_gemm_top_gb300 import ops
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    best = {}
    for method in (0, 1):
        for _ in range(3):
            ops.moe_hbm_fill(buf, 0, method)
        ms = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            ops.moe_hbm_fill(buf, 0, method)
            b.record()
            b.synchronize()
            ms.append(a.elapsed_time(b))
        best[method] = nbytes / min(ms) / 1e6
    del buf
    torch.cuda.empty_cache()
    return {"gbs": round(max(best.values()), 1), "vector_stores_gbs": round(best[0], 1),
            "bulk_copies_gbs": round(best[1], 1), "bytes": nbytes}


def memory_roofline(L, mem_ms, Rp, peaks, psrc, write_ceiling):
    """The step's memory-bound launches: algorithmic bytes (what each must
    read and write once; Rp = the rows of the 128-row-aligned groups this
    step, R = routed rows) / average CUDA-event time per launch, against
    the measured copy bandwidth, the pages' 8 TB/s and, for the write-heavy
    quantizations, the measured write-only ceiling."""
    T, d, f, R, kk = L.T, L.d, L.f, L.R, L.kk
    q = 1 + 1 / 32
    table = {
        # name: (read bytes, written bytes)
        "quant_x": (T * d * 2 + Rp * 4, 2 * Rp * d * q),
        "quant_dy": (T * d * 2 + Rp * 4 + R * 4, 2 * Rp * d * q),
        "swiglu_bwd_quant_dA": (Rp * f * 4 + Rp * 2 * f * 2, 2 * Rp * 2 * f * q),
        "combine_out": (R * d * 2 + T * kk * 8, T * d * 2),
        "combine_dx": (R * d * 2 + T * kk * 4, T * d * 2),
        "combine_bwd_dw": (T * d * 2 + R * d * 2 + T * kk * 8, T * kk * 4),
    }
    kern = {"quant_x": "k_quant_both", "quant_dy": "k_quant_both", "swiglu_bwd_quant_dA": "k_swiglu_bwd_quant",
            "combine_out": "k_combine", "combine_dx": "k_combine", "combine_bwd_dw": "k_combine_bwd"}
    out = {}
    tot_b, tot_ms = 0.0, 0.0
    for name, (rd, wr) in table.items():
        if name not in mem_ms:
            continue
        ms = mem_ms[name]
        gbs = (rd + wr) / (ms * 1e-3) / 1e9
        out[name] = {"kernel": kern[name], "ms": round(ms, 4), "read_gb": round(rd / 1e9, 3),
                     "write_gb": round(wr / 1e9, 3), "achieved_gbs": round(gbs, 1),
                     "frac_of_copy": round(gbs / peaks["hbm_gbs"], 4), "frac_of_8tbs": round(gbs / 8000.0, 4),
                     "write_gbs": round(wr / (ms * 1e-3) / 1e9, 1),
                     "frac_write_of_write_ceiling": round(wr / (ms * 1e-3) / 1e9 / write_ceiling["gbs"], 4)}
        tot_b += rd + wr
        tot_ms += ms
    agg = tot_b / (tot_ms * 1e-3) / 1e9 if tot_ms else None
    return {"bound": "hbm", "unit": "GB/s", "launches": out,
            "achieved": round(agg, 1) if agg else None, "peak": peaks["hbm_gbs"],
            "frac": round(agg / peaks["hbm_gbs"], 4) if agg else None,
            "peak_source": f"{psrc} copy bandwidth (read + write bytes)", "spec_gbs": 8000.0,
            "write_ceiling": write_ceiling, "rows_padded": Rp,
            "timing": "CUDA events around each launch in the timed eager steps, mean per launch"}


# --------------------------------------------------------------------- CPU --

def oracle_sample(workload, n_experts, seed=0):
    """Time the oracle on a bounded sample of the workload: routing of all
    tokens, then the full fwd+bwd chain (quantize, GEMMs, SwiGLU, combine
    pieces) for the routed rows of `n_experts` experts.  Returns (flops of
    the sample, seconds, description)."""
    import numpy as np
    import torch

    import oracle as O
    from grouped_gemm_top_gb300 import synth

    w = WORKLOADS[workload]
    T, d, E, k, f = w["T"], w["d"], w["E"], w["k"], w["f"]
    logits = synth.make_logits(T, E, 0, "cpu").numpy()
    x = synth.make_normal_bf16((T, d), synth.SEED_X, "cpu")
    dout = synth.make_normal_bf16((T, d), synth.SEED_DOUT, "cpu")
    rng = np.random.default_rng(seed)
    experts = rng.choice(E, size=n_experts, replace=False)
    # Expert weights are drawn directly as MXFP8 values (random E4M3 codes
    # times 2^-12), so both quantized copies of a weight equal the weight and
    # no weight quantization runs before or inside the timed region.
    wops = []
    finite = np.array([c for c in range(256) if np.isfinite(O.E4M3_VALUES[c])])
    for _ in experts:
        W1e = O.E4M3_VALUES[rng.choice(finite, size=(d, 2 * f))] * 2.0 ** -12
        W2e = O.E4M3_VALUES[rng.choice(finite, size=(f, d))] * 2.0 ** -12
        wops.append((W1e[None], W2e[None], W2e.T[None], W1e.T[None]))
    xn, dn = x.double().numpy(), dout.double().numpy()
    t0 = time.perf_counter()
    idx, wts = O.route_topk(logits, k, w["score"], w["normalize"])
    flops = 0.0
    for e, (B1, B2, B2t, B1t) in zip(experts, wops):
        tok, j = np.nonzero(idx == e)
        m = len(tok)
        if m == 0:
            continue
        offs = np.array([0, m])
        xp = xn[tok]
        q, s = O.mxfp8_quantize_rows(xp)
        A = O.grouped_gemm(O.mxfp8_dequantize_rows(q, s), B1, offs)
        h = O.bf16_round(O.swiglu(A))
        hq, hs = O.mxfp8_quantize_rows(h)
        O.grouped_gemm(O.mxfp8_dequantize_rows(hq, hs), B2, offs)
        # dy_perm as the step stores it: bf16(fp32(w * dout)) with fp32 weights
        dy = O.permute_scaled_bf16(dn, tok * k + j, k, O.fp32_round(wts))
        dq, ds = O.mxfp8_quantize_rows(dy)
        dH = O.grouped_gemm(O.mxfp8_dequantize_rows(dq, ds), B2t, offs)
        dA = O.bf16_round(O.swiglu_bwd(O.bf16_round(A), dH))
        hT, hTs, _ = O.mxfp8_quantize_cols_grouped(h, offs)
        dyT, dyTs, _ = O.mxfp8_quantize_cols_grouped(dy, offs)
        O.grouped_gemm_wgrad(O.mxfp8_dequantize_cols(hT, hTs), O.mxfp8_dequantize_cols(dyT, dyTs), offs)
        daq, das = O.mxfp8_quantize_rows(dA)
        O.grouped_gemm(O.mxfp8_dequantize_rows(daq, das), B1t, offs)
        xT, xTs, _ = O.mxfp8_quantize_cols_grouped(xp, offs)
        aT, aTs, _ = O.mxfp8_quantize_cols_grouped(dA, offs)
        O.grouped_gemm_wgrad(O.mxfp8_dequantize_cols(xT, xTs), O.mxfp8_dequantize_cols(aT, aTs), offs)
        flops += 18.0 * m * d * f
    secs = time.perf_counter() - t0
    desc = (f"routing of all {T} tokens + fwd/bwd chain (MXFP8 quantize, 6 GEMMs, SwiGLU) for the routed rows of "
            f"{n_experts} of {E} experts ({workload}); fp64 numpy")
    return flops, secs, desc


def run_gemm_point(G, M_total, NK, seed=0, steps=10, warmup=3, device="cuda:0", K=None, b_layout="gnk"):
    """Standalone grouped GEMM fwd (sweep point): G groups whose sizes are a
    Dirichlet(0.3) split of M_total rows, N = NK, K = NK (or K), A and B ~
    N(0,1) -> MXFP8, bf16 out; B in the [N][G*K] (ngk) or [G][N][K] (gnk)
    layout.  Returns a dict with TFLOPS and roofline fractions."""
    N = NK
    K = NK if K is None else K
    import numpy as np
    import torch

    from grouped_gemm_top_gb300 import ops, synth
    ops.moe_init(torch.device(device).index or 0)
    sizes = synth.dirichlet_group_sizes(G, M_total, 0.3, seed)
    gofs = np.concatenate([[0], np.cumsum((sizes + 127) // 128 * 128)])
    M = int(gofs[-1])
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=device)
    src = synth.make_normal_bf16((M_total, K), seed + 100, device)
    r = 0
    for g, m in enumerate(sizes):
        x[int(gofs[g]):int(gofs[g]) + int(m)] = src[r:r + int(m)]
        r += int(m)
    del src
    gofs_t = torch.tensor(gofs, dtype=torch.int32, device=device)
    xq, xs = ops.mxfp8_group_quantize(x, ops.MOE_QUANT_ROWWISE, gofs_t, G)
    del x
    if b_layout == "gnk":
        W = synth.make_normal_bf16((G * N, K), seed + 200, device)
        bq, bs = ops.mxfp8_group_quantize(W, ops.MOE_QUANT_ROWWISE)
        lay = ops.MOE_B_GNK
    else:
        W = synth.make_normal_bf16((G * K, N), seed + 200, device)
        wg = torch.arange(0, (G + 1) * K, K, dtype=torch.int32, device=device)
        bq, bs = ops.mxfp8_group_quantize(W, ops.MOE_QUANT_COLWISE_GROUPED, wg, G)
        lay = ops.MOE_B_NGK
    del W
    d = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)

    def launch():
        ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, xq, xs, bq, bs, lay, gofs_t, G, M, N, K, d=d, err=err)

    for _ in range(warmup):
        launch()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    assert int(err.item()) == 0, int(err.item())
    ms = sum(a.elapsed_time(b) for a, b in evs) / steps
    flops = 2.0 * M_total * N * K
    byts = G * N * K * (1 + 1 / 32) + M_total * K * (1 + 1 / 32) + M_total * N * 2
    peaks, psrc = _peaks()
    mx_peak = 2.0 * peaks["bf16_tflops"]          # kernel timed alone: burst
    t_roof = max(flops / (mx_peak * 1e12), byts / (peaks["hbm_gbs"] * 1e9))
    return {"G": G, "M_total": M_total, "N": N, "K": K, "b_layout": b_layout, "ms": round(ms, 4),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 1), "frac_flops": round(flops / (ms * 1e-3) / 1e12 / mx_peak, 4),
            "frac_roofline": round(t_roof / (ms * 1e-3), 4), "algorithmic_gb": round(byts / 1e9, 3),
            "peak_tflops": mx_peak, "peak_source": f"2 x {psrc} bf16 burst", "empty_groups": int((sizes == 0).sum())}


def run_gemm_point_nvfp4(G, M_total, N, K, seed=0, steps=10, warmup=3, device="cuda:0"):
    """Standalone NVFP4 grouped GEMM (fwd): the same Dirichlet(0.3) groups as
    run_gemm_point, A and B ~ N(0,1) quantized by nvfp4_quantize (E2M1 codes,
    UE4M3 scales per 16, fp32 tensor scales), bf16 out.  The peak is the
    measured bf16 burst rate times the nominal dense FP4/BF16 ratio
    (13.5 / 2.25 PF/s = 6)."""
    import numpy as np
    import torch

    from grouped_gemm_top_gb300 import ops, synth
    ops.moe_init(torch.device(device).index or 0)
    sizes = synth.dirichlet_group_sizes(G, M_total, 0.3, seed)
    gofs = np.concatenate([[0], np.cumsum((sizes + 127) // 128 * 128)])
    M = int(gofs[-1])
    x = torch.zeros((M, K), dtype=torch.bfloat16, device=device)
    src = synth.make_normal_bf16((M_total, K), seed + 100, device)
    r = 0
    for g, m in enumerate(sizes):
        x[int(gofs[g]):int(gofs[g]) + int(m)] = src[r:r + int(m)]
        r += int(m)
    del src
    gofs_t = torch.tensor(gofs, dtype=torch.int32, device=device)
    aq, asf, ast = ops.nvfp4_quantize(x)
    del x
    W = synth.make_normal_bf16((G * N, K), seed + 200, device)
    bq, bsf, bst = ops.nvfp4_quantize(W)
    del W
    d = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)

    def launch():
        ops.grouped_gemm_nvfp4(ops.MOE_GEMM_FWD, aq, asf, ast, bq, bsf, bst, gofs_t, G, M, N, K, d=d, err=err)

    for _ in range(warmup):
        launch()
    torch.cuda.synchronize()
    evs = []
    for _ in range(steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        launch()
        b.record()
        evs.append((a, b))
    torch.cuda.synchronize()
    assert int(err.item()) == 0, int(err.item())
    ms = sum(a.elapsed_time(b) for a, b in evs) / steps
    flops = 2.0 * M_total * N * K
    byts = G * N * K * (0.5 + 1 / 16) + M_total * K * (0.5 + 1 / 16) + M_total * N * 2
    peaks, psrc = _peaks()
    fp4_peak = 6.0 * peaks["bf16_tflops"]
    t_roof = max(flops / (fp4_peak * 1e12), byts / (peaks["hbm_gbs"] * 1e9))
    return {"format": "nvfp4", "G": G, "M_total": M_total, "N": N, "K": K, "ms": round(ms, 4),
            "tflops": round(flops / (ms * 1e-3) / 1e12, 1), "frac_flops": round(flops / (ms * 1e-3) / 1e12 / fp4_peak, 4),
            "frac_roofline": round(t_roof / (ms * 1e-3), 4), "algorithmic_gb": round(byts / 1e9, 3),
            "peak_tflops": fp4_peak, "peak_source": f"6 x {psrc} bf16 burst (nominal dense FP4/BF16 13.5/2.25)",
            "empty_groups": int((sizes == 0).sum())}


def run_wgrad_point(G, M_total, Mo, No, seed=0, steps=10, warmup=3, device="cuda:0"):
    """Standalone weight-gradient GEMM dW_g = X_g^T dY_g over Dirichlet(0.3)
    groups of M_total rows (X [rows, Mo], dY [rows, No] ~ N(0,1), rows laid
    out at 128-row group offsets), in MXFP8 (group-aware columnwise MXFP8
    operands) and in NVFP4 (group-aware columnwise NVFP4): one line with
    both.  The MXFP8 figure is the layer's own form when M is a multiple of
    256 (256 x 224 CTA-pair tiles, dY's scales in the tile-224 layout);
    `mxfp8_tile256_ms` is the 256-wide single-accumulator form beside it.
    Peaks as for the fwd points (2x / 6x the measured bf16 burst)."""
    import numpy as np
    import torch

    from grouped_gemm_top_gb300 import ops, synth
    ops.moe_init(torch.device(device).index or 0)
    sizes = synth.dirichlet_group_sizes(G, M_total, 0.3, seed)
    gofs = np.concatenate([[0], np.cumsum((sizes + 127) // 128 * 128)])
    rows = (int(gofs[-1]) + 255) // 256 * 256
    gofs_t = torch.tensor(gofs, dtype=torch.int32, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)

    def grouped(cols, sd):
        x = torch.zeros((rows, cols), dtype=torch.bfloat16, device=device)
        src = synth.make_normal_bf16((M_total, cols), sd, device)
        r = 0
        for g, m in enumerate(sizes):
            x[int(gofs[g]):int(gofs[g]) + int(m)] = src[r:r + int(m)]
            r += int(m)
        return x

    X, Y = grouped(Mo, seed + 300), grouped(No, seed + 400)
    _, _, xq8, xs8 = ops.mxfp8_gather_quantize(X, gofs_t, G, rows, None, 1, None, False, True, err=err)
    _, _, yq8, ys8 = ops.mxfp8_gather_quantize(Y, gofs_t, G, rows, None, 1, None, False, True, err=err)
    t224 = Mo % 256 == 0
    if t224:
        _, _, yq8t, ys8t = ops.mxfp8_gather_quantize(Y, gofs_t, G, rows, None, 1, None, False, True, err=err,
                                                     col_sf_layout=ops.MOE_SF_TILE224)
    xq4, xs4, xt4 = ops.nvfp4_quantize_cols(X, gofs_t, G, err=err)
    yq4, ys4, yt4 = ops.nvfp4_quantize_cols(Y, gofs_t, G, err=err)
    del X, Y
    d = torch.empty((G, Mo, No), dtype=torch.bfloat16, device=device)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        assert int(err.item()) == 0, int(err.item())
        return a.elapsed_time(b) / steps

    ms256 = timed(lambda: ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, xq8, xs8, yq8, ys8, ops.MOE_B_GNK, gofs_t, G,
                                                 Mo, No, rows, d=d, err=err))
    ms8 = ms256
    if t224:
        ms8 = timed(lambda: ops.grouped_gemm_mxfp8(ops.MOE_GEMM_WGRAD, xq8, xs8, yq8t, ys8t, ops.MOE_B_SF_TILE224,
                                                   gofs_t, G, Mo, No, rows, d=d, err=err))
    ms4 = timed(lambda: ops.grouped_gemm_nvfp4(ops.MOE_GEMM_WGRAD, xq4, xs4, xt4, yq4, ys4, yt4, gofs_t, G, Mo, No,
                                               rows, d=d, err=err))
    flops = 2.0 * M_total * Mo * No
    peaks, psrc = _peaks()
    return {"G": G, "M_total": M_total, "M": Mo, "N": No, "mxfp8_ms": round(ms8, 4),
            "mxfp8_tflops": round(flops / (ms8 * 1e-3) / 1e12, 1),
            "mxfp8_tiles": "256x224 pair, two accumulators" if t224 else "256x256 pair",
            "mxfp8_tile256_ms": round(ms256, 4), "nvfp4_ms": round(ms4, 4),
            "nvfp4_tflops": round(flops / (ms4 * 1e-3) / 1e12, 1),
            "nvfp4_frac_of_fp4_peak": round(flops / (ms4 * 1e-3) / 1e12 / (6.0 * peaks["bf16_tflops"]), 4),
            "mxfp8_frac_of_mxfp8_peak": round(flops / (ms8 * 1e-3) / 1e12 / (2.0 * peaks["bf16_tflops"]), 4),
            "output_gb": round(G * Mo * No * 2 / 1e9, 3), "peak_source": f"{psrc} bf16 burst x 2 (MXFP8) / x 6 (FP4)"}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args):
    """The oracle as it stands, timed on the host cores (bounded sample)."""
    n_exp = 1
    for _ in range(args.warmup):
        oracle_sample(args.workload, n_exp, seed=0)
    tot_f, tot_s = 0.0, 0.0
    desc = ""
    for i in range(args.steps):
        fl, s, desc = oracle_sample(args.workload, n_exp, seed=i + 1)
        tot_f += fl
        tot_s += s
    value = tot_f / tot_s / 1e12
    w = WORKLOADS[args.workload]
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot_s / args.steps, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": w["desc"], "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def max_over_ranks(ms, world, device):
    """The slowest rank's time (every rank calls this): replicas run the same
    step, and the job's step time is that of the slowest one."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step, world, ms_per_step):
    """Whole-job throughput: every replica runs one step of flops_per_step in
    the (slowest rank's) ms_per_step (weak scaling)."""
    return world * flops_per_step / (ms_per_step * 1e-3) / 1e12


def run_hbm_probe(nbytes=4 << 30, reps=10):
    """Write-only and read+write HBM bandwidth on this GPU: the library's
    own write stream (moe_hbm_fill, both methods: 16-byte vector stores and
    bulk copies out of shared memory) and a torch copy_ (read + write
    bytes).  CUDA events, 3 warm-ups, buffers of 4 GB (written) and 2 GB +
    2 GB (copied), far above L2."""
    import torch

    from grouped_gemm_top_gb300 import ops
    ops.moe_init(0)
    b = torch.empty(nbytes // 2, dtype=torch.uint8, device="cuda")
    c = torch.zeros(nbytes // 2, dtype=torch.uint8, device="cuda")

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    copy_ms = timed(lambda: b.copy_(c))
    del b, c
    wc = hbm_write_ceiling("cuda", nbytes, reps)
    peaks, src = _peaks()
    return {"write_only_gbs": wc["gbs"], "write_vector_stores_gbs": wc["vector_stores_gbs"],
            "write_bulk_copies_gbs": wc["bulk_copies_gbs"], "copy_gbs": round(nbytes / copy_ms / 1e6, 1),
            "copy_peak_file_gbs": peaks["hbm_gbs"], "peak_source": src,
            "method": "moe_hbm_fill over 4 GB (write-only, best of both methods) and torch copy_ of 2 GB into "
                      "2 GB (read+write bytes)"}


def run_seeds(args):
    """The whole step captured once in a CUDA graph and replayed over
    args.seeds routing draws (seed i: the workload's logits with seed i, so
    for the Zipf workload a different expert order and skew each time);
    only the logits buffer changes between seeds, the graph does not (the
    group sizes never reach the host).  Per seed: replay time (CUDA events
    over args.steps replays after one warm replay), the largest expert's
    share of the tokens and the number of experts with no rows.  Reports
    the median over seeds."""
    import torch

    from grouped_gemm_top_gb300 import build as _b
    if not os.path.exists(_b.LIB):
        _b.build()
    from grouped_gemm_top_gb300 import synth
    from grouped_gemm_top_gb300.layer import MoELayer

    w = WORKLOADS[args.workload]
    T, d, E, k, f = w["T"], w["d"], w["E"], w["k"], w["f"]
    dev = "cuda:0"
    stream = torch.cuda.current_stream()
    L = MoELayer(T, d, E, k, f, w["score"], w["normalize"], device=dev, wgrad224_rows=args.wgrad224_rows)
    inp = synth.make_layer_inputs(T, d, E, f, dev, zipf_s=w["zipf"])
    L.set_weights(inp["W1"], inp["W2"])
    L.x.copy_(inp["x"])
    L.dout.copy_(inp["dout"])
    L.logits.copy_(inp["logits"])
    del inp
    for _ in range(3):
        L.step_()
    L.capture()
    flops = L.flops_per_step()
    per_seed = []
    with ClockSampler(0) as clk:
        for seed in range(args.seeds):
            L.logits.copy_(synth.make_logits(T, E, synth.SEED_LOGITS + seed, dev, w["zipf"]))
            L.replay()
            torch.cuda.synchronize()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(args.steps):
                L.replay()
            s1.record(stream)
            torch.cuda.synchronize()
            L.check_err()
            counts = L.counts.cpu()
            ms = s0.elapsed_time(s1) / args.steps
            per_seed.append({"seed": seed, "ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                             "top_expert_token_share": round(int(counts.max()) / T, 4),
                             "empty_experts": int((counts == 0).sum())})
    ms_sorted = sorted(p["ms"] for p in per_seed)
    med = statistics.median(ms_sorted)
    return {"seeds": {"workload": w["desc"], "n_seeds": args.seeds, "replays_per_seed": args.steps,
                      "median_ms": round(med, 4), "median_tflops": round(flops / (med * 1e-3) / 1e12, 1),
                      "min_ms": ms_sorted[0], "max_ms": ms_sorted[-1], "per_seed": per_seed,
                      "clocks": clk.summary(), "timing": "one CUDA graph of the whole fwd+bwd step, replayed"}}


def run_compare(args, capacity_factors=(1.0, 1.25)):
    """The grouped dropless step against the prior-art ways of running the
    same layer (grouped_gemm_top_gb300.comparators): a loop of per-expert
    GEMMs with the counts read on the host every step, and capacity-based
    MoE with static padded groups (graph-captured; drops what overflows).
    Every arm is timed over args.steps steps after 3 warm-ups with CUDA
    events on the launching stream; throughput counts the dropless FLOPs
    18 T k d f for every arm, so padding and dropped tokens both show as
    lost throughput."""
    import torch

    from grouped_gemm_top_gb300 import build as _b
    if not os.path.exists(_b.LIB):
        _b.build()
    from grouped_gemm_top_gb300 import synth
    from grouped_gemm_top_gb300.comparators import CapacityMoE, LoopMoE
    from grouped_gemm_top_gb300.layer import MoELayer

    w = WORKLOADS[args.workload]
    T, d, E, k, f = w["T"], w["d"], w["E"], w["k"], w["f"]
    dev = "cuda:0"
    stream = torch.cuda.current_stream()
    inp = synth.make_layer_inputs(T, d, E, f, dev, zipf_s=w["zipf"])

    def load(L):
        L.set_weights(inp["W1"], inp["W2"])
        L.logits.copy_(inp["logits"])
        L.x.copy_(inp["x"])
        L.dout.copy_(inp["dout"])

    def timed(fn, steps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record(stream)
        for _ in range(steps):
            fn()
        e.record(stream)
        torch.cuda.synchronize()
        return s.elapsed_time(e) / steps

    flops = 18.0 * T * k * d * f

    def arm(ms, **kw):
        return dict(ms_per_step=round(ms, 4), tflops=round(flops / (ms * 1e-3) / 1e12, 1), **kw)

    arms = {}
    L = MoELayer(T, d, E, k, f, w["score"], w["normalize"], device=dev)
    load(L)
    per_step = KERNELS_PER_STEP + (WGRAD_SPLIT_KERNELS if L.wgrad_split else 0)
    arms["grouped_dropless_eager"] = arm(timed(L.step_, args.steps), launches_per_step=per_step)
    L.capture()
    arms["grouped_dropless_graph"] = arm(timed(L.replay, args.steps), launches_per_step=per_step)
    L.check_err()
    counts = L.counts.cpu()
    L.graph = None
    loop = LoopMoE(L)
    loop.set_weights(inp["W1"], inp["W2"])
    ms = timed(loop.step_, max(2, args.steps // 3))
    L.check_err()
    arms["loop_of_gemms"] = arm(ms, launches_per_step=loop.launches, host_syncs_per_step=1,
                                note="counts copied to the host and synchronised every step; one GEMM per expert")
    del loop, L
    torch.cuda.empty_cache()
    for cf in capacity_factors:
        C = CapacityMoE(T, d, E, k, f, w["score"], w["normalize"], device=dev, capacity_factor=cf)
        load(C)
        C.capture()
        ms = timed(C.replay, args.steps)
        C.check_err()
        arms[f"capacity_cf{cf}_graph"] = arm(ms, capacity_rows_per_expert=C.C, computed_rows=E * C.C,
                                            routed_rows=T * k, dropped_fraction=round(C.dropped_fraction(), 5))
        del C
        torch.cuda.empty_cache()
    return {"compare": {"workload": w["desc"], "flops_per_step_dropless": flops, "steps": args.steps,
                        "max_expert_rows": int(counts.max()), "mean_expert_rows": T * k / E, "arms": arms}}


def run_vendor_point(M, N, K, steps=10, warmup=3, device="cuda:0"):
    """One dense MXFP8 GEMM D[M,N] = A[M,K] B[N,K]^T (bf16 out) timed two
    ways on the same E4M3 codes: the library's block-scaled GEMM
    (torch._scaled_mm with E8M0 scales per 32, which calls cuBLASLt) and our
    grouped GEMM with one group.  This is context for the grouped kernel's
    roofline fraction: the rate a vendor GEMM reaches on this GPU for the
    same contraction.  The library's scales are all 1.0 (the values do not
    change the time); A is larger than L2, so no flush is needed."""
    import torch

    from grouped_gemm_top_gb300 import ops, synth
    ops.moe_init(torch.device(device).index or 0)
    a = synth.make_normal_bf16((M, K), 1, device)
    aq, asf = ops.mxfp8_group_quantize(a, ops.MOE_QUANT_ROWWISE)
    del a
    b = synth.make_normal_bf16((N, K), 2, device)
    bq, bsf = ops.mxfp8_group_quantize(b, ops.MOE_QUANT_ROWWISE)
    del b
    gofs = torch.tensor([0, M], dtype=torch.int32, device=device)
    d = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(steps):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / steps

    flops = 2.0 * M * N * K
    peaks, psrc = _peaks()
    mx_peak = 2.0 * peaks["bf16_tflops"]
    out = {"M": M, "N": N, "K": K, "peak_tflops": mx_peak, "peak_source": f"2 x {psrc} bf16 burst"}
    ms = timed(lambda: ops.grouped_gemm_mxfp8(ops.MOE_GEMM_FWD, aq, asf, bq, bsf, ops.MOE_B_GNK, gofs, 1,
                                              M, N, K, d=d, err=err))
    assert int(err.item()) == 0, int(err.item())
    out["ours"] = {"ms": round(ms, 4), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
    try:
        def round_up(v, m):
            return (v + m - 1) // m * m
        sa = torch.full((round_up(M, 128) * round_up(K // 32, 4),), 127, dtype=torch.uint8, device=device)
        sb = torch.full((round_up(N, 128) * round_up(K // 32, 4),), 127, dtype=torch.uint8, device=device)
        sa, sb = sa.view(torch.float8_e8m0fnu), sb.view(torch.float8_e8m0fnu)
        A8, B8 = aq.view(torch.float8_e4m3fn), bq.view(torch.float8_e4m3fn).t()   # B column-major [K, N]
        ms = timed(lambda: torch._scaled_mm(A8, B8, sa, sb, out_dtype=torch.bfloat16))
        out["library"] = {"call": "torch._scaled_mm (cuBLASLt, MXFP8 1x32)", "ms": round(ms, 4),
                          "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
        out["ours_over_library"] = round(out["library"]["ms"] / out["ours"]["ms"], 3)
    except Exception as e:          # the installed torch may not offer MXFP8 _scaled_mm
        out["library"] = {"unavailable": f"{type(e).__name__}: {str(e).splitlines()[0][:200]}"}
    out["frac_ours"] = round(out["ours"]["tflops"] / mx_peak, 4)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="deepseek-v3", choices=sorted(WORKLOADS))
    ap.add_argument("--router", action="store_true",
                    help="include the router (logits = x W_r, bf16 tensor-core GEMMs, and its backward) in the "
                         "step and report its GEMMs separately")
    ap.add_argument("--shared-experts", type=int, default=0, metavar="S",
                    help="add S shared experts (every token, weight 1) as extra groups of the same grouped GEMMs")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-experts", type=int, default=6)
    ap.add_argument("--gemm-point", nargs="+", type=int, metavar="G M_TOTAL N [K]",
                    help="time one standalone grouped GEMM fwd (K = N unless given) and print its line")
    ap.add_argument("--b-layout", default="gnk", choices=["ngk", "gnk"])
    ap.add_argument("--wgrad-point", nargs=4, type=int, metavar=("G", "M_TOTAL", "M", "N"),
                    help="time the weight-gradient grouped GEMM in MXFP8 and in NVFP4 and print one line")
    ap.add_argument("--nvfp4", action="store_true",
                    help="with --gemm-point / --sweep: the NVFP4 grouped GEMM (E2M1, UE4M3 scales per 16) instead")
    ap.add_argument("--sweep", action="store_true", help="the 18-point grouped GEMM sweep, one line per point")
    ap.add_argument("--wgrad224-rows", type=int, nargs=2, default=None, metavar=("LO", "HI"),
                    help="only groups of LO <= rows < HI (HI 0: unbounded) take 224-wide weight-gradient tiles, "
                         "the rest 256-wide ones (0 0: all 224; default: the layer's WGRAD224_ROWS)")
    ap.add_argument("--seeds", type=int, default=0, metavar="S",
                    help="replay the captured step over S routing seeds (e.g. --workload deepseek-v3-zipf "
                         "--seeds 20) and print the median; one line")
    ap.add_argument("--compare", action="store_true",
                    help="time the grouped dropless step against a per-expert GEMM loop and capacity-based MoE on "
                         "the same workload and print one line")
    ap.add_argument("--vendor-point", nargs=3, type=int, metavar=("M", "N", "K"),
                    help="time one dense MXFP8 GEMM with the library's block-scaled GEMM (torch._scaled_mm) and "
                         "with ours (one group) and print one line")
    ap.add_argument("--hbm-probe", action="store_true",
                    help="measure write-only (moe_hbm_fill) and copy (torch copy_) HBM bandwidth and print one line")
    args = ap.parse_args()
    if args.hbm_probe:
        print(json.dumps({"hbm_probe": run_hbm_probe()}), flush=True)
        return
    if args.compare:
        print(json.dumps(run_compare(args)), flush=True)
        return
    if args.vendor_point:
        print(json.dumps({"vendor_point": run_vendor_point(*args.vendor_point, steps=args.steps,
                                                           warmup=max(args.warmup, 3))}), flush=True)
        return
    if args.seeds:
        print(json.dumps(run_seeds(args)), flush=True)
        return
    if args.wgrad_point:
        G, Mt, Mo, No = args.wgrad_point
        with ClockSampler(0) as clk:
            r = run_wgrad_point(G, Mt, Mo, No, steps=args.steps, warmup=max(args.warmup, 3))
        r["clocks"] = clk.summary()
        print(json.dumps({"wgrad_point": r}), flush=True)
        return
    if args.gemm_point or args.sweep:
        if args.gemm_point:
            gp = list(args.gemm_point)
            pts = [(gp[0], gp[1], gp[2], gp[3] if len(gp) > 3 else gp[2])]
        else:
            pts = [(G, M, NK, NK) for G in (8, 64, 256) for NK in (2048, 7168) for M in (16384, 65536, 262144)]
        for i, (G, M, N, K) in enumerate(pts):
            with ClockSampler(0) as clk:
                if args.nvfp4:
                    r = run_gemm_point_nvfp4(G, M, N, K, seed=i, steps=args.steps, warmup=max(args.warmup, 3))
                else:
                    r = run_gemm_point(G, M, N, seed=i, steps=args.steps, warmup=max(args.warmup, 3), K=K,
                                       b_layout=args.b_layout)
            r["clocks"] = clk.summary()
            print(json.dumps({"sweep_point": r}), flush=True)
            import torch
            torch.cuda.empty_cache()
        return
    args.warmup = max(args.warmup, 3) if args.impl == "ours" else args.warmup

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    result, L = run_gpu(args, rank, world, local_rank)
    del L
    if rank == 0:
        if not args.no_cpu_baseline:
            fl, secs, desc = oracle_sample(args.workload, args.cpu_experts)
            result["cpu_baseline"] = {"value": round(fl / secs / 1e12, 6), "unit": "TFLOPS", "cores": cpu_cores(),
                                      "kind": "oracle", "sample": desc, "seconds": round(secs, 2)}
        else:
            result["cpu_baseline"] = None
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

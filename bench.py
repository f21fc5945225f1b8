#!/usr/bin/env python
"""Benchmark: W4A16 GEMV achieved HBM GB/s and % of the GB300 roofline.

One step = one token's decode layer stack of a dense 9B-class decoder at
M = 1: 36 layers x (q 4096x4096, k/v 1024x4096, o 4096x4096, gate+up
24576x4096, down 4096x12288) plus a 151936x4096 lm_head, W4A16 affine g64,
each projection with its own bf16 activation vector (217 GEMV launches,
4.27 GB of weights, scales, activations and outputs), issued as one CUDA graph.
`value` = algorithmic bytes of the step / step time (inputs resident in HBM;
the 4.27 GB working set is 33x the L2, so every step streams from HBM).

Also reported in the same JSON line: the M = 16 stack (skinny form), the MXFP4
MoE layer at T = 1 and 16, the block-32 Hadamard + int8 path and the W8A8
int32 GEMM at 4096x4096 / 12288x4096, the single 1024x1024 GEMV, the
end-to-end number through the public API with host buffers, the roofline of
the dominant kernel, the CPU baseline (the oracle on the host cores) and the
SM clocks sampled during the timed region.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica of the stack ("replicas
only": the path has no exchange step); value = bytes of all ranks / max time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "W4A16 GEMV achieved HBM GB/s and % of GB300 peak at M=1 and M=16"
FALLBACK_HBM = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extras", action="store_true", help="only the M=1 stack")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--case", default=None, help="run one kernel case a few times (for ncu): " + ", ".join(CASES))
    ap.add_argument("--reps", type=int, default=3)
    return ap.parse_args()


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(t, world, device):
    """The job's step time: the largest per-rank time over all ranks."""
    tmax = torch.tensor([float(t)], device=device, dtype=torch.float64)
    if world > 1:
        torch.distributed.all_reduce(tmax, op=torch.distributed.ReduceOp.MAX)
    return float(tmax.item())


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 0.0)), "measured"
    return FALLBACK_HBM, 1900.0, "fallback"


def w4_bytes(N, K, M=1):
    return N * K // 2 + 2 * N * (K // 64) * 2 + M * (K * 2 + N * 4)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        inside = [r for r in rows if self.t0 and self.t1 and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        use = inside if inside else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for i, n in enumerate(names):
                if r[3][5 + i].lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use), "in_timed_region": bool(inside)}


# --------------------------------------------------------------------------- helpers

def capture(graph_fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        graph_fn()
    return g


def replay_timed(g, iters, stream, warmup=2):
    """Replay `g` on `stream` (warm-up, then `iters` timed replays bracketed by
    CUDA events on the same stream); seconds per replay."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / iters * 1e-3


def time_graph(graph_fn, iters, stream):
    g = capture(graph_fn, stream)
    return replay_timed(g, iters, stream), g


def build_stack(q, dev, M, layers=36, seed=1):
    """Weights of the layer stack (4.26 GB) plus per-projection inputs."""
    shapes = synth.stack_layer_shapes(layers)
    mats = []
    for i, (name, N, K) in enumerate(shapes):
        wq, s, b = synth.w4_weights(N, K, seed=seed, slot=10 + i, device=dev)
        mats.append((name, N, K, wq, s, b))
    return mats


def stack_io(mats, dev, M, seed=1):
    xs, ys = [], []
    for i, (name, N, K, *_r) in enumerate(mats):
        xs.append(synth.bf16_normal((M, K), seed=seed, slot=5000 + i, device=dev))
        ys.append(torch.empty(M, N, device=dev, dtype=torch.float32))
    return xs, ys


def prime_skinny_workspace(q, mats, M, dev, stream):
    """Allocate (outside any capture) the zero-filled skinny workspace every
    projection of the stack will share on `stream`."""
    need = max(q.lib().qg_skinny_workspace_size(M, N, K, 64) for (_, N, K, *_r) in mats)
    if need:
        q.skinny_workspace(need, dev, stream)


def run_stack(q, mats, xs, ys, M, stream):
    for (name, N, K, wq, s, b), x, y in zip(mats, xs, ys):
        if M == 1:
            q.qgemv_w4a16(wq, s, b, x[0], y[0], stream=stream)
        else:
            q.qgemm_w4a16_skinny(wq, s, b, x, y, stream=stream)


def kernel_traffic(kind, alg_bytes_avg):
    """Per-launch DRAM traffic from the committed ncu summary, scaled to the
    average launch of the step; None if the kernel source changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kind)
    if not d:
        return None
    src = os.path.join(ROOT, d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != d["source_sha256"]:
        return None
    return d["dram_bytes_per_alg_byte"] * alg_bytes_avg


# --------------------------------------------------------------------------- CPU baseline

def cpu_sample_stack(div, seed=1):
    """Every projection of the stack with ceil(N/div) rows (rows are i.i.d.)."""
    out = []
    for i, (name, N, K) in enumerate(synth.stack_layer_shapes()):
        n = max(1, -(-N // div))
        wq, s, b = synth.w4_weights(n, K, seed=seed + 100, slot=i)
        x = synth.bf16_normal((1, K), seed=seed + 100, slot=5000 + i)
        out.append((n, K, wq.numpy().view("uint32"), s.view(torch.int16).numpy().view("uint16"),
                    b.view(torch.int16).numpy().view("uint16"), x.view(torch.int16).numpy().view("uint16")))
    return out


def run_cpu_sample(sample, budget_s=None):
    import oracle
    t0 = time.perf_counter()
    nbytes = 0
    done = 0
    for (n, K, wq, s, b, x) in sample:
        oracle.w4a16(wq, s, b, x)
        nbytes += w4_bytes(n, K)
        done += 1
        if budget_s is not None and time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return nbytes, dt, done


def cpu_baseline(seconds, mats=None, xs=None, stride=8):
    """The oracle on the host cores over every `stride`-th row of every
    projection of the stack (rows copied from the device-resident weights),
    repeated until `seconds` of CPU time have elapsed."""
    import oracle
    oracle.build()
    if mats is None:
        sample = cpu_sample_stack(16)
    else:
        sample = []
        for (name, N, K, wq, s, b), x in zip(mats, xs):
            sel = torch.arange(0, N, stride, device=wq.device)
            sample.append((len(sel), K, wq[sel].cpu().numpy().view("uint32"),
                           s[sel].cpu().view(torch.int16).numpy().view("uint16"),
                           b[sel].cpu().view(torch.int16).numpy().view("uint16"),
                           x[:1].cpu().view(torch.int16).numpy().view("uint16")))
    nbytes, dt, passes, done = 0, 0.0, 0, 0
    while dt < seconds:
        b, t, d = run_cpu_sample(sample, budget_s=seconds - dt)
        nbytes += b
        dt += t
        done += d
        passes += 1
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"float64 C oracle, every {stride}th output row of all 217 stack projections "
                      f"({done} projection passes, {nbytes / 1e6:.0f} MB of algorithmic bytes in {dt:.1f} s)"}


def reference_arm(args, rank, world):
    if rank != 0:
        return
    import oracle
    oracle.build()
    div = 64
    sample = cpu_sample_stack(div)
    for _ in range(args.warmup):
        run_cpu_sample(sample[:6])
    total_b, total_t = 0, 0.0
    for _ in range(args.steps):
        b, t, _ = run_cpu_sample(sample)
        total_b += b
        total_t += t
    v = total_b / total_t / 1e9
    sample_desc = (f"each step: the float64 C oracle over all 217 projections of the stack with rows cut to "
                   f"ceil(N/{div}) ({total_b / args.steps / 1e6:.0f} MB of algorithmic bytes)")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_t / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode layer stack, 9B-class dense, W4A16 g64, M=1 (row-sampled)"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": sample_desc},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- extras

def bench_single_gemv(q, dev, stream, l2_bytes):
    N = K = 1024
    per = w4_bytes(N, K)
    copies = max(8, (4 * l2_bytes) // per + 1)
    mats = [synth.w4_weights(N, K, seed=0, slot=i, device=dev) for i in range(copies)]
    x = synth.bf16_normal((K,), 0, 99999, dev)
    y = torch.empty(N, device=dev)

    def fn():
        for wq, s, b in mats:
            q.qgemv_w4a16(wq, s, b, x, y, stream=stream)
    t, _ = time_graph(fn, 5, stream)
    t /= copies
    return {"us_per_call": t * 1e6, "GB_per_s": per / t / 1e9, "weight_copies_rotated": int(copies)}


def bench_w8a16(q, dev, stream, hbm_peak):
    """The row-int8 output head, 151936 x 4096 (622 MB of weights > L2)."""
    N, K = 151936, 4096
    wq, s = synth.w8_row_weights(N, K, seed=3, slot=1, device=dev)
    x = synth.bf16_normal((K,), 3, 2, dev)
    y = torch.empty(N, device=dev)
    t, _ = time_graph(lambda: q.qgemv_w8a16(wq, s, x, y, stream=stream), 20, stream)
    nbytes = N * K + 4 * N + 2 * K + 4 * N
    del wq, s
    return {"us_per_call": t * 1e6, "GB_per_s": nbytes / t / 1e9, "frac": nbytes / t / 1e9 / hbm_peak,
            "algorithmic_bytes": nbytes}


def bench_affine(q, dev, stream, hbm_peak):
    """qgemm_affine at M = 1 on the lm_head shape (151936 x 4096, > L2 at every
    width): codes at 2, 3, 4, 5, 6 and 8 bits with groups of 64, and 4 bits with
    groups of 32 and 128 (the chunked kernel; the 4-bit g64 case has the W4A16
    fast path)."""
    N, K = 151936, 4096
    x = synth.bf16_normal((K,), 3, 2, dev)
    y = torch.empty(N, device=dev)
    out = {}
    for bits, group in ((2, 64), (3, 64), (4, 64), (5, 64), (6, 64), (8, 64), (4, 32), (4, 128)):
        wq, s, b = synth.affine_weights(N, K, bits, 5, bits, device=dev, group=group)
        t, _ = time_graph(lambda: q.qgemm_affine(wq, bits, s, b, x, y=y, stream=stream), 10, stream)
        nbytes = N * K * bits // 8 + 4 * N * (K // group) + 2 * K + 4 * N
        out[f"b{bits}_g{group}"] = {"us_per_call": t * 1e6, "GB_per_s": nbytes / t / 1e9,
                                   "frac": nbytes / t / 1e9 / hbm_peak, "algorithmic_bytes": nbytes}
        del wq, s, b
    return out


def bench_skinny_stacks(q, mats, dev, stream, hbm_peak):
    """The layer stack at M in {2, 4, 8, 16, 32} activation rows (continuous-batch
    rows or speculative-tree tokens): one grouped skinny launch per step
    (warp-level MMA up to 16 rows, tcgen05 above)."""
    out = {}
    for M in (2, 4, 8, 16, 32):
        xsM, ysM = stack_io(mats, dev, M)
        step = sum(w4_bytes(N, K, M) for (_, N, K, *_r) in mats)
        grp = q.SkinnyGroup([(wq, s, b, x, y) for (_, N, K, wq, s, b), x, y in zip(mats, xsM, ysM)])
        t, _ = time_graph(lambda: grp.run(stream), 10, stream)
        grp.close()
        form = "one grouped skinny launch over the 217 projections"
        out[f"M{M}"] = {"value": step / t / 1e9, "unit": "GB/s", "frac": step / t / 1e9 / hbm_peak,
                        "ms_per_step": t * 1e3, "tokens_per_s": M / t, "bytes_per_step": step, "form": form}
        del xsM, ysM
    return out


def decoder_chain_items(q, mats, x0, dev):
    """The decode step of the dense stack in dependency order: per layer
    {q, k, v} at level 4l reading the layer input, o reading q's output (the
    stand-in for attention), gate_up reading o's output, down reading the gate
    half of gate_up's output; the next layer and the lm_head read down's
    output. Every input is a copy scaled by 1 / (0.02 sqrt(K_src)) (the
    weights' std is 0.02) in place of the norm layers, so the activations stay
    O(1) through the 36 layers (a fixed-scale SwiGLU would square them every
    layer)."""
    items, level, layer_in, by = [], 0, (q.X_BF16, x0, 1.0), {}
    for name, N, K, wq, s, b in mats:
        kind = name.split(".")[-1]
        y = torch.empty(N, device=dev)
        if kind in ("q", "k", "v", "lm_head"):
            (op, x, alpha), lvl = layer_in, level
        elif kind == "o":
            op, x, alpha, lvl = q.X_COPY, by["q"], 1.0 / (0.02 * 64.0), level + 1
        elif kind == "gate_up":
            op, x, alpha, lvl = q.X_COPY, by["o"], 1.0 / (0.02 * 64.0), level + 2
        else:
            op, x, alpha, lvl = q.X_COPY, by["gate_up"], 1.0 / (0.02 * 64.0), level + 3
        items.append(dict(wq=wq, scales=s, biases=b, level=lvl, op=op, x=x, alpha=alpha, y=y))
        by[kind] = y
        if kind == "down":
            level += 4
            layer_in = (q.X_COPY, y, 1.0 / (0.02 * 12288 ** 0.5))
    return items


def bench_dependent_stack(q, mats, dev, stream, hbm_peak, steps):
    """The M = 1 stack in dependency order (145 levels: per layer {q, k, v}, o,
    gate_up, down; then lm_head) as one chain launch per token, and the same
    217 projections as one level (all independent) through the same kernel."""
    step_bytes = sum(w4_bytes(N, K) for (_, N, K, *_r) in mats)
    x0 = synth.bf16_normal((4096,), 1, 4999, device=dev)
    out = {}
    for key, one_level in (("dependent_stack_m1", False), ("chain_one_level_m1", True)):
        items = decoder_chain_items(q, mats, x0, dev)
        if one_level:
            xs = [synth.bf16_normal((it["wq"].shape[1] * 8,), 1, 6000 + i, device=dev) for i, it in enumerate(items)]
            for it, x in zip(items, xs):
                it.update(level=0, op=q.X_BF16, x=x, alpha=1.0)
        ch = q.GemvChain(items)
        g = capture(lambda: ch.run(stream), stream)
        reps = []
        for _ in range(5):
            reps.append(replay_timed(g, max(20, steps), stream, warmup=3))
        reps.sort()
        t = reps[len(reps) // 2]
        assert q.device_error() == 0
        levels = items[-1]["level"] + 1
        out[key] = {"value": step_bytes / t / 1e9, "unit": "GB/s", "frac": step_bytes / t / 1e9 / hbm_peak,
                    "traffic": kernel_traffic("w4a16_chain_m1", step_bytes),
                    "ms_per_step": t * 1e3, "tokens_per_s": 1.0 / t, "bytes_per_step": step_bytes,
                    "levels": levels, "launches_per_step": 1,
                    "min_ms_per_step": reps[0] * 1e3, "max_ms_per_step": reps[-1] * 1e3,
                    "form": ("one w4a16_chain_kernel launch per token; per layer {q, k, v} -> o -> gate_up -> "
                             "down -> next layer, each level awaited in the kernel" if not one_level else
                             "the 217 projections as one level of the same chain kernel (independent inputs)")}
        del g
        ch.close()
        del items
        torch.cuda.empty_cache()
    return out


def bench_moe(q, dev, stream, T, moe_w):
    E, H, I, k = 384, 7168, 2048, 16
    x = synth.bf16_normal((T, H), 3, 0, dev)
    lg = synth.router_logits(T, E, 3, 1, dev)
    ws = torch.empty(q.moe_workspace_size(T, H, I, E, k), dtype=torch.uint8, device=dev)
    y = torch.empty(T, H, device=dev)
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    wt = torch.empty(T, k, device=dev)

    def fn():
        q.moe_mxfp4_expert_forward(x, lg, *moe_w, top_k=k, y=y, topk_idx=idx, topk_w=wt, workspace=ws,
                                   stream=stream)
    t, _ = time_graph(fn, 20, stream)
    D = int(torch.unique(idx).numel())
    per_expert = 3 * (H * I // 2 + H * I // 32)
    nbytes = D * per_expert + T * (2 * H + 4 * E + 4 * H)
    return {"us_per_call": t * 1e6, "GB_per_s": nbytes / t / 1e9, "distinct_experts": D,
            "algorithmic_bytes": nbytes}


def bench_w8a8(q, dev, stream, N, l2_bytes):
    K, M = 4096, 16
    wf = synth.normal_f32((N, K), 0.02, 4, 20, dev).to(torch.bfloat16)
    sb = synth.sign_bits(K, 4, 5, dev)
    wq, _ = q.hadamard32_quant_i8(wf, sb)
    copies = max(4, (4 * l2_bytes) // (N * K) + 1)
    ws = [wq.clone() for _ in range(copies)]
    xa = synth.outlier_activations(M, K, 4, 0, dev)
    qa, sa = q.hadamard32_quant_i8(xa, sb)
    c = torch.empty(M, N, dtype=torch.int32, device=dev)

    def fn():
        for w in ws:
            q.gemm_w8a8_i32(qa, w, c, stream=stream)
    t, _ = time_graph(fn, 5, stream)
    t /= copies
    nbytes = N * K + M * K + M * N * 4

    def fh():
        for _ in range(50):
            q.hadamard32_quant_i8(xa, sb, qa, sa, stream=stream)
    th, _ = time_graph(fh, 3, stream)
    # the fused path: transform + int8 + product + dequant in one launch (y fp32)
    _, swq = q.hadamard32_quant_i8(wf, sb)
    y = torch.empty(M, N, device=dev)
    q.gemm_w8a8_hadamard(xa, sb, ws[0], swq, y, stream=stream)  # workspace allocated outside the capture

    def ff():
        for w in ws:
            q.gemm_w8a8_hadamard(xa, sb, w, swq, y, stream=stream)
    tf, _ = time_graph(ff, 5, stream)
    tf /= copies
    fbytes = N * K + 4 * N + 2 * M * K + 4 * M * N
    return {"us_per_call": t * 1e6, "GB_per_s": nbytes / t / 1e9, "weight_copies_rotated": int(copies),
            "hadamard_quant_us_per_call": th / 50 * 1e6,
            "two_launch_path_us": (t + th / 50) * 1e6,
            "fused": {"us_per_call": tf * 1e6, "GB_per_s": fbytes / tf / 1e9, "algorithmic_bytes": fbytes,
                      "form": "gemm_w8a8_hadamard: one cooperative launch, x bf16 -> y fp32"}}


# --------------------------------------------------------------------------- single cases (profiling)

CASES = ["gemv_lm_head", "gemv_down", "gemv_q", "skinny16_gate_up", "skinny16_down", "moe_T1", "moe_T16",
         "w8a16_lm_head",
         "w8a8_12288", "hadamard_16x4096", "gemv_group_4layers", "skinny16_group_4layers", "chain_4layers",
         "chain_flat_4layers", "chain_trace", "w8a8_fused_12288", "w8a8_fused_4096",
         "skinny32_group_4layers", "skinny8_group_4layers", "affine_b4_lm_head", "affine_b6_lm_head"]


def chain_trace_summary(q, dev):
    """The dependency-ordered chain of the full stack with its level trace on:
    per level kind (q/k/v, o, gate_up, down, lm_head) the mean over layers of
    the level's duration (previous level's last publish to this one's) and of
    its parts, medians over the CTAs: release (previous level complete -> this
    CTA's wait ends), build (wait end -> input fragments built) and tiles
    (built -> the CTA's last publish), plus the slowest CTA's tiles."""
    mats = build_stack(q, dev, 1)
    x0 = synth.bf16_normal((4096,), 1, 4999, device=dev)
    ch = q.GemvChain(decoder_chain_items(q, mats, x0, dev))
    for _ in range(3):
        ch.run()
    ch.trace(True)
    ch.run()
    torch.cuda.synchronize()
    tr = ch.trace_read().astype(np.float64)
    ch.close()
    tr[tr == 0] = np.nan
    tr = (tr - np.nanmin(tr)) / 1e3  # us
    done = np.nanmax(tr[:, :, 3], axis=0)
    L = tr.shape[1]
    kinds = ["qkv", "o", "gate_up", "down"]
    rows = {}
    for l in range(1, L):
        k = kinds[l % 4] if l < L - 1 else "lm_head"
        prev = done[l - 1]
        wait_end, built, pub = tr[:, l, 1], tr[:, l, 2], tr[:, l, 3]
        built = np.where(np.isnan(built), wait_end, built)
        r = rows.setdefault(k, {"n": 0, "level_us": 0.0, "release_us": 0.0, "build_us": 0.0, "tiles_us": 0.0,
                                "tiles_max_us": 0.0})
        r["n"] += 1
        r["level_us"] += done[l] - prev
        r["release_us"] += np.nanmedian(wait_end - prev)
        r["build_us"] += np.nanmedian(built - wait_end)
        r["tiles_us"] += np.nanmedian(pub - built)
        r["tiles_max_us"] += np.nanmax(pub - built)
    out = {k: {f: (round(v / r["n"], 2) if f != "n" else v) for f, v in r.items()} for k, r in rows.items()}
    out["total_us"] = round(float(np.nanmax(tr)), 1)
    return out


def run_case(args):
    """One kernel on one full-size (or, for the MoE, reduced-E) input; warm-up
    launches then `reps` launches. Small device footprint, for ncu captures."""
    import skinny_gemm_qgemv_gb300 as q
    q.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    c = args.case
    if c == "chain_trace":
        print(json.dumps(chain_trace_summary(q, dev)), flush=True)
        return
    if c == "gemv_group_4layers":
        # the grouped launch over 4 decoder layers + the lm_head (0.78 GB)
        mats = build_stack(q, dev, 1, layers=4)
        xs, ys = stack_io(mats, dev, 1)
        grp = q.GemvGroup([(wq, s, b, x[0], y[0]) for (_, N, K, wq, s, b), x, y in zip(mats, xs, ys)])
        f = grp.run
        nbytes = sum(w4_bytes(N, K) for (_, N, K, *_r) in mats)
    elif c in ("chain_4layers", "chain_flat_4layers"):
        # the dependent-order chain over 4 decoder layers + the lm_head (0.78 GB, 17 levels),
        # or the same projections as one level with independent inputs
        mats = build_stack(q, dev, 1, layers=4)
        x0 = synth.bf16_normal((4096,), 1, 4999, device=dev)
        items = decoder_chain_items(q, mats, x0, dev)
        if c == "chain_flat_4layers":
            for i, it in enumerate(items):
                it.update(level=0, op=q.X_BF16, x=synth.bf16_normal((it["wq"].shape[1] * 8,), 1, 6000 + i, device=dev))
        ch = q.GemvChain(items)
        f = ch.run
        nbytes = sum(w4_bytes(N, K) for (_, N, K, *_r) in mats)
    elif c in ("skinny8_group_4layers", "skinny16_group_4layers", "skinny32_group_4layers"):
        # the grouped skinny launch over 4 decoder layers + the lm_head: M = 8
        # or 16 (warp-level MMA kernel, one or two n tiles) or M = 32 (tcgen05 kernel)
        Mr = int(c[6:8].rstrip("_"))
        mats = build_stack(q, dev, Mr, layers=4)
        xs, ys = stack_io(mats, dev, Mr)
        grp = q.SkinnyGroup([(wq, s, b, x, y) for (_, N, K, wq, s, b), x, y in zip(mats, xs, ys)])
        f = grp.run
        nbytes = sum(w4_bytes(N, K, Mr) for (_, N, K, *_r) in mats)
    elif c.startswith("gemv_") or c.startswith("skinny16_"):
        shape = {"lm_head": (151936, 4096), "down": (4096, 12288), "q": (4096, 4096),
                 "gate_up": (24576, 4096)}[c.split("_", 1)[1]]
        M = 1 if c.startswith("gemv_") else 16
        N, K = shape
        wq, s, b = synth.w4_weights(N, K, 1, 0, dev)
        x = synth.bf16_normal((M, K), 1, 1, dev)
        y = torch.empty(M, N, device=dev)
        f = (lambda: q.qgemv_w4a16(wq, s, b, x[0], y[0])) if M == 1 else \
            (lambda: q.qgemm_w4a16_skinny(wq, s, b, x, y))
        nbytes = w4_bytes(N, K, M)
    elif c.startswith("moe_"):
        T = int(c[5:])
        E, H, I, k = 64, 7168, 2048, 16
        gq, gs = synth.mxfp4_weights(E * I, H, 3, 2, dev)
        uq, us = synth.mxfp4_weights(E * I, H, 3, 3, dev)
        dq, ds = synth.mxfp4_weights(E * H, I, 3, 4, dev)
        w = [t.reshape(E, r, -1) for t, r in ((gq, I), (gs, I), (uq, I), (us, I), (dq, H), (ds, H))]
        x = synth.bf16_normal((T, H), 3, 0, dev)
        lg = synth.router_logits(T, E, 3, 1, dev)
        f = lambda: q.moe_mxfp4_expert_forward(x, lg, *w, top_k=k)  # noqa: E731
        nbytes = None
    elif c.startswith("affine_b"):
        # qgemm_affine at M = 1 on the lm_head shape, 4 or 6-bit codes, groups of 64
        bits = int(c[8])
        N, K = 151936, 4096
        wq, s, b = synth.affine_weights(N, K, bits, 5, bits, device=dev, group=64)
        x = synth.bf16_normal((K,), 3, 2, dev)
        y = torch.empty(N, device=dev)
        f = lambda: q.qgemm_affine(wq, bits, s, b, x, y=y)  # noqa: E731
        nbytes = N * K * bits // 8 + 4 * N * (K // 64) + 2 * K + 4 * N
    elif c == "w8a16_lm_head":
        N, K = 151936, 4096
        wq, s = synth.w8_row_weights(N, K, 3, 1, dev)
        x = synth.bf16_normal((K,), 3, 2, dev)
        y = torch.empty(N, device=dev)
        f = lambda: q.qgemv_w8a16(wq, s, x, y)  # noqa: E731
        nbytes = N * K + 8 * N + 2 * K
    elif c == "w8a8_12288":
        N, K = 12288, 4096
        a = torch.randint(-127, 128, (16, K), dtype=torch.int8, device=dev)
        w = torch.randint(-127, 128, (N, K), dtype=torch.int8, device=dev)
        f = lambda: q.gemm_w8a8_i32(a, w)  # noqa: E731
        nbytes = N * K + 16 * K + 16 * N * 4
    elif c.startswith("w8a8_fused_"):
        N, K, M = int(c.split("_")[-1]), 4096, 16
        wf = synth.normal_f32((N, K), 0.02, 4, 20, dev).to(torch.bfloat16)
        sb = synth.sign_bits(K, 4, 5, dev)
        wq, swq = q.hadamard32_quant_i8(wf, sb)
        xa = synth.outlier_activations(M, K, 4, 0, dev)
        y = torch.empty(M, N, device=dev)
        f = lambda: q.gemm_w8a8_hadamard(xa, sb, wq, swq, y)  # noqa: E731
        nbytes = N * K + 4 * N + 2 * M * K + 4 * M * N
    elif c == "hadamard_16x4096":
        x = synth.outlier_activations(16, 4096, 4, 0, dev)
        sb = synth.sign_bits(4096, 4, 5, dev)
        f = lambda: q.hadamard32_quant_i8(x, sb)  # noqa: E731
        nbytes = 16 * 4096 * 3
    else:
        raise SystemExit(f"unknown case {c}")
    for _ in range(3):
        f()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.reps):
        f()
    e1.record()
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / args.reps
    print(json.dumps({"case": c, "us_per_call": t * 1e6,
                      "GB_per_s": None if nbytes is None else nbytes / t / 1e9}), flush=True)
    assert q.device_error() == 0


# --------------------------------------------------------------------------- main

def main():
    args = parse()
    if args.case:
        return run_case(args)
    rank, world, local = dist_info()
    if world > 1 and not torch.distributed.is_initialized():
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        reference_arm(args, rank, world)
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    import skinny_gemm_qgemv_gb300 as q
    q.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    hbm_peak, _, peak_src = peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    q.set_pdl(True)

    # ---------------- config: the M = 1 layer stack
    with torch.cuda.stream(stream):
        mats = build_stack(q, dev, 1)
        xs, ys = stack_io(mats, dev, 1)
    torch.cuda.synchronize()
    step_bytes = sum(w4_bytes(N, K) for (_, N, K, *_r) in mats)
    launches = len(mats)

    # The step as one persistent grouped launch over the 217 projections (each
    # has its own activation vector, so they are independent); the same step
    # as 217 separate launches is measured below for comparison.
    grp = q.GemvGroup([(wq, s, b, x[0], y[0]) for (_, N, K, wq, s, b), x, y in zip(mats, xs, ys)])
    g = capture(lambda: grp.run(stream), stream)
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            g.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    # The K-step timed region is repeated (each repeat exactly K steps, events
    # on the replaying stream) until about 0.6 s of timed work, at least 5
    # times, so the clock sampler covers it; the value is the median repeat.
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    rep_times = []
    clocks.mark("t0")
    while len(rep_times) < 5 or (sum(rep_times) < 0.6 and len(rep_times) < 200):
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        rep_times.append(e0.elapsed_time(e1) * 1e-3)
    torch.cuda.synchronize()
    clocks.mark("t1")
    if world > 1:
        torch.distributed.barrier()
    reps_sorted = sorted(rep_times)
    t_step = reps_sorted[len(reps_sorted) // 2] / args.steps
    repeats = {"n": len(rep_times), "steps_each": args.steps, "min_ms_per_step": reps_sorted[0] / args.steps * 1e3,
               "median_ms_per_step": t_step * 1e3, "max_ms_per_step": reps_sorted[-1] / args.steps * 1e3}
    time.sleep(0.25)
    clocks.stop()
    t_step = max_over_ranks(t_step, world, dev)
    value = world * step_bytes / t_step / 1e9

    # ---------------- the same step as 217 launches (one per projection) in one graph
    g217 = capture(lambda: run_stack(q, mats, xs, ys, 1, stream), stream)
    t217 = replay_timed(g217, max(20, min(args.steps, 500)), stream)
    del g217

    # ---------------- roofline of the dominant kernel: the step is one launch of
    # w4a16_group_kernel (the graph has no other node), so its launch duration
    # is the event-timed step time. Per-shape durations of the per-projection
    # kernel come from graphs holding the 36 launches of one projection kind.
    per_shape = {}
    for kind in ("q", "k", "o", "gate_up", "down", "lm_head"):
        sel = [i for i, m in enumerate(mats) if m[0].split(".")[-1] == kind]
        gk = capture(lambda: run_stack(q, [mats[i] for i in sel], [xs[i] for i in sel], [ys[i] for i in sel],
                                       1, stream), stream)
        tk = replay_timed(gk, 10, stream) / len(sel)
        N, K = mats[sel[0]][1], mats[sel[0]][2]
        per_shape[kind] = {"N": N, "K": K, "us_per_launch": tk * 1e6, "GB_per_s": w4_bytes(N, K) / tk / 1e9}
        del gk
    k_time = t_step
    achieved = step_bytes / k_time / 1e9
    traffic = kernel_traffic("w4a16_group_m1", step_bytes)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak, "traffic": traffic,
                "kernel": "w4a16_group_kernel (one launch per step over the 217 projections)",
                "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)" if peak_src == "measured"
                else "fallback 6.8 TB/s",
                "avg_launch_us": k_time * 1e6, "alg_bytes_per_launch": step_bytes,
                "per_launch_form": {"kernel": "w4a16_gemv_kernel<1, ...>", "launches_per_step": launches,
                                    "GB_per_s": world * step_bytes / t217 / 1e9,
                                    "frac": step_bytes / t217 / 1e9 / hbm_peak, "ms_per_step": t217 * 1e3,
                                    "per_shape": per_shape}}

    # ---------------- e2e through the public API with host buffers
    xh = torch.empty(sum(x.numel() for x in xs), dtype=torch.bfloat16).pin_memory()
    yh = torch.empty(sum(y.numel() for y in ys), dtype=torch.float32).pin_memory()
    xd = torch.empty(xh.numel(), dtype=torch.bfloat16, device=dev)
    yd = torch.empty(yh.numel(), dtype=torch.float32, device=dev)
    xv, yv, o1, o2 = [], [], 0, 0
    for x, y in zip(xs, ys):
        xv.append(xd[o1:o1 + x.numel()].view_as(x))
        yv.append(yd[o2:o2 + y.numel()].view_as(y))
        o1 += x.numel()
        o2 += y.numel()
    xh.copy_(torch.cat([x.reshape(-1) for x in xs]).cpu())

    grp_e2e = q.GemvGroup([(wq, s, b, x[0], y[0]) for (_, N, K, wq, s, b), x, y in zip(mats, xv, yv)])

    def e2e_step():
        xd.copy_(xh, non_blocking=True)
        grp_e2e.run(stream)
        yh.copy_(yd, non_blocking=True)
    ge = capture(e2e_step, stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            ge.replay()
        stream.synchronize()
        n_e2e = max(10, min(args.steps, 500))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            ge.replay()
            stream.synchronize()
        t_e2e = (time.perf_counter() - t0) / n_e2e
    e2e = {"value": world * step_bytes / t_e2e / 1e9, "unit": "GB/s", "h2d_bytes_per_step": xh.numel() * 2,
           "d2h_bytes_per_step": yh.numel() * 4,
           "how": "pinned host x -> device, one C-ABI grouped GEMV run over the 217 projections, device y -> "
                  "pinned host, one CUDA graph per step, host-timed including the final synchronize"}

    extras = {}
    if not args.no_extras and rank == 0:
        # M = 16 stack (skinny form), same weights
        xs16, ys16 = stack_io(mats, dev, 16)
        step16 = sum(w4_bytes(N, K, 16) for (_, N, K, *_r) in mats)
        grp16 = q.SkinnyGroup([(wq, s, b, x, y) for (_, N, K, wq, s, b), x, y in zip(mats, xs16, ys16)])
        t16, _ = time_graph(lambda: grp16.run(stream), 20, stream)
        prime_skinny_workspace(q, mats, 16, dev, stream)
        t16s, _ = time_graph(lambda: run_stack(q, mats, xs16, ys16, 16, stream), 20, stream)
        extras["m16_stack"] = {"value": step16 / t16 / 1e9, "unit": "GB/s", "frac": step16 / t16 / 1e9 / hbm_peak,
                               "ms_per_step": t16 * 1e3, "tokens_per_s": 16 / t16, "bytes_per_step": step16,
                               "form": "one grouped skinny launch (B-fragment pass + warp-level MMA kernel) over the 217 projections",
                               "per_launch_form": {"value": step16 / t16s / 1e9, "unit": "GB/s",
                                                   "frac": step16 / t16s / 1e9 / hbm_peak,
                                                   "ms_per_step": t16s * 1e3}}
        grp16.close()
        del xs16, ys16, grp16
        extras["skinny_stack"] = bench_skinny_stacks(q, mats, dev, stream, hbm_peak)
        extras.update(bench_dependent_stack(q, mats, dev, stream, hbm_peak, args.steps))
        extras["m1_stack_tokens_per_s"] = 1.0 / t_step
        extras["single_gemv_1024"] = bench_single_gemv(q, dev, stream, l2)
        extras["w8a16_lm_head_151936x4096"] = bench_w8a16(q, dev, stream, hbm_peak)
        extras["affine_m1_151936x4096"] = bench_affine(q, dev, stream, hbm_peak)
        torch.cuda.empty_cache()
        E, H, I = 384, 7168, 2048
        with torch.cuda.stream(stream):
            gq, gs = synth.mxfp4_weights(E * I, H, 3, 2, dev)
            uq, us = synth.mxfp4_weights(E * I, H, 3, 3, dev)
            dq, ds = synth.mxfp4_weights(E * H, I, 3, 4, dev)
        moe_w = [t.reshape(E, r, -1) for t, r in ((gq, I), (gs, I), (uq, I), (us, I), (dq, H), (ds, H))]
        torch.cuda.synchronize()
        for T in (1, 16, 32):  # the two configured batches, then 32 (the largest of the same kernels)
            r = bench_moe(q, dev, stream, T, moe_w)
            r["frac"] = r["GB_per_s"] / hbm_peak
            extras[f"moe_mxfp4_T{T}"] = r
        del moe_w, gq, gs, uq, us, dq, ds
        torch.cuda.empty_cache()
        for N in (4096, 12288):
            r = bench_w8a8(q, dev, stream, N, l2)
            r["frac"] = r["GB_per_s"] / hbm_peak
            r["fused"]["frac"] = r["fused"]["GB_per_s"] / hbm_peak
            extras[f"w8a8_{N}x4096"] = r

    cpu = cpu_baseline(args.cpu_seconds, mats, xs) if rank == 0 else None
    assert q.device_error() == 0, "a kernel reported a bounded-wait timeout"

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "decode layer stack of a dense 9B-class decoder, M=1: 36 x (q, k, v, o, "
                                   "gate+up, down) + lm_head 151936x4096, W4A16 affine g64, 217 GEMVs per step",
                       "bytes_per_step": step_bytes, "gemvs_per_step": launches,
                       "issue": "one persistent grouped launch over the 217 independent projections (each with "
                                "its own activation vector); roofline.per_launch_form has the same step as 217 "
                                "launches",
                       "l2": f"inputs {step_bytes / 1e9:.2f} GB > L2 {l2 / 1e6:.0f} MB (no flush needed)",
                       "parallelism": f"replicas x{world}", "frac_of_peak": value / world / hbm_peak,
                       "tokens_per_s": world / t_step},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks.summary(),
            "repeats": repeats, "gpu_launches": args.steps * repeats["n"], "extras": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Throughput of the multi-tenant LoRA delta on one GB300 (per GPU replica).

One step = one pass of the hot path over one batch: device metadata build
(stable sort of tokens by adapter) + the fused shrink/expand of every packed
slice (dense workloads), or metadata + MoE w13 + MoE w2 (MoE workloads).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl gb300|reference]

Prints one JSON line.  Under torchrun every rank runs its own replica on its
own GPU (the path shards by token with no exchange step: "replicas only"),
the timed region is bracketed by a barrier and a device synchronise, and the
time is the maximum over ranks.
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
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from heterogeneous_adapters_lora_gb300 import inputs as gen  # noqa: E402

WORKLOADS = {
    "decode_qkv": "decode BGMV, Llama-3-8B packed QKV: T=256 (1 token/request), H=4096 -> 4096/1024/1024, "
                  "32 adapters rank 16, idx uniform over 32 + 10% -1, scale 2",
    "tiny": "single 512 -> 512 projection, T=64, 4 adapters rank 8, idx over {-1,0..3}, scale 2",
    "prefill_gate_up": "prefill SGMV gate_up: 8 requests, lengths U[128,2048] contiguous, H=4096 -> 2x14336, "
                       "8 adapters rank 64, request i -> adapter i",
    "prefill_r16": "prefill SGMV gate_up as 'prefill_gate_up' with rank 16 (the tensor-core path below rank 64)",
    "many_adapter_down": "many-adapter decode down_proj 14336 -> 4096, T=2048, 1024 adapters ranks {8,16,32,64} "
                         "padded to 64, Zipf(1.2) popularity",
    "moe": "MoE-LoRA: E=64, top-8 of softmax(N(0,1)), D=2048, F=1408, 8 adapters rank 16, T=1024, "
           "w13 (gate+up) and w2",
    "moe_shared": "MoE-LoRA as 'moe' in the shared-outer layout (w13-A and w2-B expert dim 1)",
    "moe_decode": "MoE-LoRA at decode: as 'moe' with T=16 (128 pairs over 512 (adapter, expert) keys: "
                  "sparse occupancy, one 16-row tile per non-empty key)",
    "moe_sparse": "MoE-LoRA at sparse occupancy: as 'moe' with T=8 (64 pairs, T*top_k*8 = 512 <= 64 experts x "
                  "8 adapters: the regime of the pages' naive block assignment)",
    "linear_qkv": "full LoRA linear layer at decode: the decode_qkv batch with its base weight 4096 -> 6144 "
                  "and bias: y = x W^T + bias (cuBLASLt) + LoRA delta",
    "linear_prefill": "full LoRA linear layer at prefill: the prefill_gate_up batch (~8K tokens in 8 contiguous "
                      "runs, rank 64) with its base weight 4096 -> 2x14336: y = x W^T + LoRA delta",
    "inkling_sink": "Inkling sink experts at decode: T=256, d_model 2048, 2 sink experts of d_mlp 1408: "
                    "w13 LoRA (2048 -> 2x2816) + SiLU(gate)*up*gamma + w2 LoRA (2816 -> 2048), "
                    "8 adapters rank 16, scale 2, 10% -1",
}


def make_case(name):
    if name == "decode_qkv":
        return gen.decode_qkv()
    if name == "tiny":
        return gen.tiny()
    if name == "prefill_gate_up":
        return gen.prefill_gate_up()
    if name == "prefill_r16":
        return gen.prefill_gate_up(rank=16)
    if name == "many_adapter_down":
        return gen.many_adapter_down()
    if name == "moe":
        return gen.moe()
    if name == "moe_shared":
        return gen.moe(shared_outer=True)
    if name == "moe_decode":
        return gen.moe(T=16)
    if name == "moe_sparse":
        return gen.moe(T=8)
    if name == "inkling_sink":
        return gen.inkling_sink()
    if name == "linear_qkv":
        return gen.linear_qkv()
    if name == "linear_prefill":
        return gen.linear_prefill()
    raise ValueError(name)


def is_moe(name):
    return name.startswith("moe")


def is_sink(name):
    return name == "inkling_sink"


def is_linear(name):
    return name.startswith("linear_")


def is_plain_dense(name):
    return not (is_moe(name) or is_sink(name) or is_linear(name))


def do_step(name, r):
    """One step of the hot path: a plain dense layer builds the batch metadata
    and applies the delta through the single call that does both
    (lora_build_meta_apply); the other workloads make their calls in order."""
    if is_plain_dense(name):
        r.step_batch()
    else:
        r.step()


def apply_kernels(name, policy, fused=False):
    """The kernels one apply call launches for this workload (the roofline's
    'dominant kernel': the apply's launches, timed together)."""
    if fused:
        return ("bgmv_fused_kernel in batch mode (one launch: one thread-block cluster per adapter slot does the "
                "shrink, the DSMEM reduction and the expand, one more CTA builds the batch metadata)")
    if is_moe(name):
        c = make_case(name)
        sparse = c.T * c.K * 8 <= c.E * c.L
        if policy == 5 or (policy == 0 and sparse):
            return "moe_block_kernel over the metadata's 16-row tiles (one thread-block cluster per tile) for w13 and w2"
        if policy == 4:
            return "moe_align_padded_kernel (block_m 1) + moe_block_kernel (one cluster per pair) for w13 and w2"
    if policy == 1:
        k = "grouped_lora_kernel (persistent split-K)"
    elif policy == 2:
        k = "cluster_lora_kernel (one pass, cluster DSMEM reduction)"
    else:
        expand = ("bgmv_expand_kernel (warp-level MMAs)" if policy == 8 else
                  "bgmv_expand_tc_kernel (tcgen05; bgmv_expand_kernel where a slice width is not a multiple of 128)")
        k = ("split shrink (bgmv_shrink_slot_kernel key-major, or bgmv_shrink_kernel / bgmv_shrink_tile_kernel "
             "per tile) + " + expand + ", chained by programmatic dependent launch")
    if is_sink(name):
        return k + " on w13, sink_act_kernel, the same on w2"
    if is_linear(name):
        if policy == 6:
            return ("linear_slot_kernel + the split shrink (bgmv_shrink_*) + linear_lora_kernel (tcgen05 GEMM whose "
                    "accumulator also takes the delta as extra K blocks)")
        return ("cuBLASLt base GEMM, then lora_apply_slices (bgmv_fused_kernel for decode batches, the sgmv "
                "and split kernels otherwise)")
    if name in ("prefill_gate_up", "prefill_r16") and policy != 1:
        k = "sgmv_shrink_kernel + sgmv_expand_kernel (tcgen05, 128-row runs); short tiles: " + k
    return k + (" for w13 and w2" if is_moe(name) else "")


# ----------------------------------------------------------------- algorithmic bytes

def dense_algorithmic_bytes(c):
    """Bytes of x, A, B and y the delta must touch: x rows and y rows (read +
    write) of active tokens, A and B of each distinct active slot at its true
    rank, plus the idx vector the metadata reads."""
    act = np.array([0 <= a < c.L and c.enabled[a] and c.ranks[a] > 0 for a in c.idx], bool)
    n = int(act.sum())
    slots = np.unique(c.idx[act])
    r = c.ranks[slots].astype(np.int64)
    A = int(r.sum()) * c.H * 2 * c.n_slices
    B = int(r.sum()) * c.out_total * 2
    return dict(x=n * c.H * 2, A=A, B=B, y=2 * n * c.out_total * 2, idx=c.T * 4,
                total=n * c.H * 2 + A + B + 2 * n * c.out_total * 2 + c.T * 4, active=n)


def sink_algorithmic_bytes(c):
    """w13 apply + activation (gate_up read, h written, gammas) + w2 apply
    (its x rows are h rows)."""
    a13 = dense_algorithmic_bytes(c.w13)
    a2 = dense_algorithmic_bytes(c.w2)
    W = c.n_experts * c.d_mlp
    act = c.T * (2 * W * 2 + W * 2 + c.n_experts * 4)
    total = a13["total"] + act + a2["total"] - a2["idx"]
    return dict(total=total, idx=a13["idx"], active=a13["active"], act=act)


def linear_algorithmic_bytes(c):
    """Base GEMM (W, x rows, y rows written) plus the delta's bytes."""
    a = dense_algorithmic_bytes(c)
    gemm = c.out_total * c.H * 2 + c.T * c.H * 2 + c.T * c.out_total * 2 + c.out_total * 2
    return dict(total=a["total"] + gemm, idx=a["idx"], active=a["active"], gemm=gemm)


def moe_algorithmic_bytes(c):
    t = np.repeat(np.arange(c.T), c.K)
    a = c.idx[t]
    e = c.topk_ids.reshape(-1)
    act = (a >= 0) & (a < c.L)
    act[act] &= (c.enabled[a[act]] != 0) & (c.ranks[a[act]] > 0)
    n_pairs = int(act.sum())
    tokens = np.unique(t[act])
    keys = np.unique(a[act] * c.E + e[act])
    slots = np.unique(a[act])
    r_key = c.ranks[keys // c.E].astype(np.int64)
    r_slot = c.ranks[slots].astype(np.int64)
    ea = r_slot.sum() if c.shared_outer else r_key.sum()
    w13 = (len(tokens) * c.D * 2 + c.n13 * ea * c.D * 2 + c.n13 * r_key.sum() * c.F13 * 2
           + 2 * n_pairs * c.n13 * c.F13 * 2)
    eb = r_slot.sum() if c.shared_outer else r_key.sum()
    w2 = (n_pairs * c.F * 2 + r_key.sum() * c.F * 2 + eb * c.D * 2 + 2 * n_pairs * c.D * 2 + n_pairs * 4)
    meta = c.T * 4 + c.T * c.K * 4
    return dict(w13=int(w13), w2=int(w2), meta=meta, total=int(w13 + w2 + meta), active=len(tokens),
                pairs=n_pairs)


# ----------------------------------------------------------------- clocks

CLOCK_Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
           "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
           "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- reference arm (oracle on CPU)

def oracle_step_fn(name, c):
    import oracle
    if is_moe(name):
        def step():
            oracle.moe_meta(c.topk_ids, c.idx, c.L, c.E, c.enabled, c.ranks)
            oracle.moe_w13(c)
            oracle.moe_w2(c)
        return step, c.T
    if is_linear(name):
        bias = gen.f32_to_bf16_bits(np.random.default_rng(7).normal(0, 0.5, c.out_total).astype(np.float32))
        n = 64   # bounded sample: the first 64 tokens (the oracle's base product is per token)
        from types import SimpleNamespace
        sub = SimpleNamespace(**{k: getattr(c, k) for k in ("H", "L", "R", "ranks", "scales", "enabled", "A", "B",
                                                             "out_dims", "out_total", "n_slices")})
        sub.x, sub.idx, sub.y0, sub.T = c.x[:n], c.idx[:n], c.y0[:n], n

        def step():
            oracle.dense_meta(sub.idx, c.L, c.enabled, c.ranks)
            oracle.linear(sub, c.W, bias)
        return step, n
    if is_sink(name):
        from heterogeneous_adapters_lora_gb300.inputs import f32_to_bf16_bits

        def step():
            oracle.dense_meta(c.w13.idx, c.w13.L, c.w13.enabled, c.w13.ranks)
            y13, _ = oracle.dense_delta(c.w13)
            h = oracle.sink_act(f32_to_bf16_bits(y13), c.gammas, c.n_experts, c.d_mlp)
            oracle.dense_delta(c.w2, x=h)
        return step, c.T
    if name == "many_adapter_down":
        # bounded sample: the first 256 tokens (the oracle is per-token)
        n = 256
        sub = dict(x=c.x[:n], idx=c.idx[:n], y_in=c.y0[:n])

        def step():
            oracle.dense_meta(sub["idx"], c.L, c.enabled, c.ranks)
            oracle.dense_delta(c, **sub)
        return step, n
    if name == "prefill_gate_up":
        n = 512
        sub = dict(x=c.x[:n], idx=c.idx[:n], y_in=c.y0[:n])

        def step():
            oracle.dense_meta(sub["idx"], c.L, c.enabled, c.ranks)
            oracle.dense_delta(c, **sub)
        return step, n

    def step():
        oracle.dense_meta(c.idx, c.L, c.enabled, c.ranks)
        oracle.dense_delta(c)
    return step, c.T


def cpu_sample_desc(name, c, tokens):
    if tokens == c.T:
        return f"the full batch ({c.T} tokens) per call"
    return f"the first {tokens} of {c.T} tokens per call (the oracle is per-token)"


def time_oracle(name, c, min_seconds=2.0, max_calls=1000):
    import oracle
    step, tokens = oracle_step_fn(name, c)
    step()  # build + warm
    n, t0 = 0, time.perf_counter()
    while True:
        step()
        n += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or n >= max_calls:
            break
    return dict(value=tokens * n / el, unit="tokens/s", cores=oracle.max_threads(), kind="oracle",
                sample=f"{n} oracle calls on {cpu_sample_desc(name, c, tokens)} of {name}")


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    c = make_case(args.workload)
    import oracle
    step, tokens = oracle_step_fn(args.workload, c)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = tokens * args.steps / el
    line = {"impl": "reference", "metric": "LoRA-delta tokens/s", "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {WORKLOADS[args.workload]}",
                       "sample": cpu_sample_desc(args.workload, c, tokens)},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.max_threads(),
                             "kind": "oracle", "sample": cpu_sample_desc(args.workload, c, tokens)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- GPU arm

def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "heterogeneous_adapters_lora_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, fn), "rb") as f:
                h.update(fn.encode())
                h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """dram bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    ent = rec.get(workload, {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


def load_tensor_peak():
    """Sustained dense bf16 TFLOP/s of this GPU (a kernel timed inside a long run)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except (OSError, ValueError, KeyError):
        return 1700.0, "fallback"


def linear_flops(c):
    """Algorithmic FLOPs of the full linear layer: the base GEMM over every
    token plus the shrink and expand of the tokens with an active adapter."""
    delta = sum(2 * int(c.ranks[a]) * (c.H * len(c.out_dims) + c.out_total) for a in c.idx
                if 0 <= a < c.L and c.enabled[a] and c.ranks[a] > 0)
    return 2 * c.T * c.H * c.out_total + delta


def max_over_ranks(values, world, device=None):
    """Element-wise maximum of per-rank timings (all ranks get the result)."""
    if world <= 1:
        return list(values)
    import torch
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_throughput(tokens_per_step, steps, world, ms):
    """Tokens of every replica over the slowest rank's time (weak scaling)."""
    return tokens_per_step * steps * world / (ms * 1e-3)


# workloads of the per_workload block: one per configuration of the task
# (tiny, decode QKV, prefill gate_up, many-adapter down_proj, MoE in both
# layouts), each timed like the headline
PER_WORKLOAD = ["tiny", "decode_qkv", "prefill_gate_up", "many_adapter_down", "moe", "moe_shared"]


def build_runs(name, c, dev, l2, max_copies, Hn):
    """Resident copies of the workload (pool, inputs, outputs, metadata,
    workspace), enough that their algorithmic bytes exceed twice the L2."""
    moe, sink, lin = is_moe(name), is_sink(name), is_linear(name)
    ab = (moe_algorithmic_bytes(c) if moe else sink_algorithmic_bytes(c) if sink
          else linear_algorithmic_bytes(c) if lin else dense_algorithmic_bytes(c))
    n_rot = min(max(1, math.ceil(2 * l2 / max(ab["total"], 1))), max_copies)
    bias = (gen.f32_to_bf16_bits(np.random.default_rng(7).normal(0, 0.5, c.out_total).astype(np.float32))
            if lin else None)

    def one():
        return (Hn.MoERun(c, device=dev) if moe else Hn.SinkRun(c, device=dev) if sink
                else Hn.LinearRun(c, bias, device=dev) if lin else Hn.DenseRun(c, device=dev))
    return [one() for _ in range(n_rot)], ab, one


def time_graph(torch, stream, body, reps=1):
    """Capture body() once as a CUDA graph, replay it once untimed, then time
    reps replays between CUDA events on the launching stream (ms per replay)."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        body()
    g.replay()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / reps, g


def measure(name, runs, ab, args, torch, stream, L, world, dev, sampler=None):
    """Step time (one CUDA graph of exactly args.steps steps over the rotating
    copies, timed once after its untimed first replay), the apply alone and the
    metadata build alone (graphs of KA calls), and kernel launches per step."""
    moe = is_moe(name)
    n_rot = len(runs)
    for r in runs:                       # warm-up outside any graph
        for _ in range(max(1, args.warmup)):
            do_step(name, r)
    stream.synchronize()
    n0 = L.lora_kernel_launch_count()
    do_step(name, runs[0])
    stream.synchronize()
    launches_per_step = L.lora_kernel_launch_count() - n0
    # a plain dense step of one launch is the fused kernel in batch mode
    fused = is_plain_dense(name) and launches_per_step == 1

    def steps(k):
        for i in range(k):
            do_step(name, runs[i % n_rot])

    # warm-up steps (W >= 3) as a graph, then the clocks are sampled over ~1 s
    # of the same work, and the K timed steps run while they are still sampled
    gw = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gw, stream=stream):
        steps(max(3, args.warmup))
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk, stream=stream):
        steps(args.steps)
    gw.replay()
    gk.replay()
    stream.synchronize()
    if sampler is not None:
        t_end = time.perf_counter() + args.clock_seconds
        while time.perf_counter() < t_end:
            gw.replay()
            stream.synchronize()
    gw.replay()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    gk.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    ms = e0.elapsed_time(e1)

    # the apply kernels alone (metadata built beforehand) and the metadata alone
    for r in runs:
        r.build_meta()
    KA = max(1, min(args.kernel_launches, 64))
    reps = max(1, args.kernel_launches // KA)

    def applies():
        for k in range(KA):
            r = runs[k % n_rot]
            if moe:
                r.w13()
                r.w2()
            elif fused:
                r.step_batch()  # the step's one kernel
            else:
                r.apply()

    def metas():
        for k in range(KA):
            runs[k % n_rot].build_meta()
    kms, _ = time_graph(torch, stream, applies, reps)
    meta_ms, _ = time_graph(torch, stream, metas, reps)
    return dict(ms=ms, kms=kms / KA, meta_ms=meta_ms / KA, launches_per_step=launches_per_step, n_rot=n_rot,
                fused=fused)


def kernel_bytes(name, ab, fused=False):
    """Algorithmic bytes of the timed kernels: the apply's (x, A, B, y), plus
    the idx vector when the metadata build runs in the same launch."""
    if is_moe(name):
        return ab["w13"] + ab["w2"]
    return ab["total"] if fused else ab["total"] - ab["idx"]


def run_gpu(args, rank, world, local_rank):
    import torch
    from heterogeneous_adapters_lora_gb300 import harness as Hn
    from heterogeneous_adapters_lora_gb300 import lora as L

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    L.lib()
    L.lora_set_kernel_policy(args.kernel_policy)
    name = args.workload
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    peak, peak_kind = load_peaks()
    stream = torch.cuda.Stream(device=dev)

    c = make_case(name)
    moe, sink, lin = is_moe(name), is_sink(name), is_linear(name)
    with torch.cuda.stream(stream):
        runs, ab, make_run = build_runs(name, c, dev, l2, args.max_copies, Hn)
        torch.cuda.synchronize(dev)
        with ClockSampler(local_rank) as cs:
            m = measure(name, runs, ab, args, torch, stream, L, world, dev, sampler=cs)
        ms, kms, meta_ms = m["ms"], m["kms"], m["meta_ms"]

        # end to end through the public API with host buffers: every step copies
        # its inputs in from pinned host memory, makes the calls and copies its
        # result out.  As a serving loop does, consecutive steps are pipelined
        # over three sets of device buffers: step i's copy in (one copy
        # stream), earlier steps' calls (the compute stream) and copies out (a
        # second copy stream) run at the same time; a buffer set is refilled
        # only once its previous result has been copied out.
        NSET = 3  # buffer sets: a step's copy in waits for the copy out of the step NSET back
        e_runs = [runs[q] if len(runs) > q else make_run() for q in range(NSET)]

        # the step's inputs (attribute paths on a run) and their host arrays;
        # the outputs are copied back from the run's tensors
        if moe:
            in_paths = ["x", "ic2", "idx", "topk", "topk_w", "ic1", "ic3"]
            h_arrays = [c.x.view(np.int16), c.ic2.view(np.int16), c.idx, c.topk_ids, c.topk_w.reshape(-1),
                        c.ic1_0.view(np.int16), c.ic3_0.view(np.int16)]
            out_paths = ["ic1", "ic3"]
        elif lin:
            in_paths, h_arrays, out_paths = ["x", "idx"], [c.x.view(np.int16), c.idx], ["y"]
        elif sink:
            in_paths = ["r13.x", "r13.idx", "r13.y", "gammas", "r2.y"]
            h_arrays = [c.w13.x.view(np.int16), c.w13.idx, c.w13.y0.view(np.int16), c.gammas, c.w2.y0.view(np.int16)]
            out_paths = ["r2.y"]
        else:
            in_paths, h_arrays, out_paths = ["x", "idx", "y"], [c.x.view(np.int16), c.idx, c.y0.view(np.int16)], ["y"]

        def attr(r, path):
            o = r
            for k in path.split(".")[:-1]:
                o = getattr(o, k)
            return o, path.split(".")[-1]

        # Inputs staged as a serving loop would: one pinned host buffer and,
        # per buffer set, one device buffer of the same layout whose pieces are
        # the run's input tensors (views), so a step copies its inputs in with
        # a single copy (each copy costs a few microseconds of its own).
        offs, size = [], 0
        for a in h_arrays:
            offs.append(size)
            size = (size + np.ascontiguousarray(a).nbytes + 255) // 256 * 256
        h_pack = torch.empty(size, dtype=torch.uint8).pin_memory()
        for a, o in zip(h_arrays, offs):
            b = np.ascontiguousarray(a).view(np.uint8).reshape(-1)
            h_pack[o:o + b.size].copy_(torch.from_numpy(b))
        d_packs = []
        for r in e_runs:
            buf = torch.empty(size, dtype=torch.uint8, device=dev)
            for pth, o in zip(in_paths, offs):
                obj, k = attr(r, pth)
                t = getattr(obj, k)
                v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                v.copy_(t)
                setattr(obj, k, v)
            d_packs.append(buf)

        def io(r):
            return [getattr(*attr(r, pth)) for pth in out_paths]

        h_out = [[torch.empty_like(d, device="cpu").pin_memory() for d in io(r)] for r in e_runs]
        bi = size
        bo = sum(t.numel() * t.element_size() for t in h_out[0])
        s_in = torch.cuda.Stream(device=dev)
        s_out = torch.cuda.Stream(device=dev)

        def e2e_steps(n):
            """n pipelined steps; every stream joins the current one at the end."""
            ev_in = [torch.cuda.Event() for _ in range(n)]
            ev_calls = [torch.cuda.Event() for _ in range(n)]
            ev_out = [torch.cuda.Event() for _ in range(n)]
            start = torch.cuda.Event()
            start.record(stream)
            s_in.wait_event(start)
            s_out.wait_event(start)
            for i in range(n):
                b = i % NSET
                r = e_runs[b]
                d_out = io(r)
                if i >= NSET:
                    s_in.wait_event(ev_out[i - NSET])  # set b's last result is out, its calls done
                with torch.cuda.stream(s_in):
                    d_packs[b].copy_(h_pack, non_blocking=True)
                    ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                with torch.cuda.stream(stream):
                    do_step(name, r)
                    ev_calls[i].record(stream)
                s_out.wait_event(ev_calls[i])
                with torch.cuda.stream(s_out):
                    for h, d in zip(h_out[b], d_out):
                        h.copy_(d, non_blocking=True)
                    ev_out[i].record(s_out)
            stream.wait_event(ev_in[n - 1])
            stream.wait_event(ev_out[n - 1])

        for _ in range(max(1, args.warmup)):
            e2e_steps(2)
        stream.synchronize()
        # the pipelined steps captured as one CUDA graph of G steps (pinned-memory
        # copies and the cross-stream waits are graph nodes), replayed
        G = 16
        e2e_graph = None
        try:
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge, stream=stream):
                e2e_steps(G)
            ge.replay()
            stream.synchronize()
            e2e_graph = ge
        except Exception:  # capture not supported here: time the eager calls
            e2e_graph = None
            torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        reps = max(1, -(-args.steps // G))
        e2e_n = reps * G
        f0.record(stream)
        for _ in range(reps):
            if e2e_graph is not None:
                e2e_graph.replay()
            else:
                e2e_steps(G)
        f1.record(stream)
        stream.synchronize()
        e2e_ms = f0.elapsed_time(f1)
        for r in runs + e_runs[1:]:
            r.close()
        del runs, e_runs
        torch.cuda.synchronize(dev)

        # every other configuration of the task, timed the same way (step graph
        # of exactly K steps, the apply and the metadata alone)
        per = {}
        if not args.no_per_workload and world == 1:
            for wn in PER_WORKLOAD:
                if wn == name:
                    continue
                wc = make_case(wn)
                w_runs, w_ab, _ = build_runs(wn, wc, dev, l2, args.max_copies, Hn)
                torch.cuda.synchronize(dev)
                wm = measure(wn, w_runs, w_ab, args, torch, stream, L, world, dev)
                for r in w_runs:
                    r.close()
                del w_runs
                torch.cuda.synchronize(dev)
                wkb = kernel_bytes(wn, w_ab, wm["fused"])
                ent = {"tokens_per_s": wc.T * args.steps / (wm["ms"] * 1e-3), "step_us": wm["ms"] / args.steps * 1e3,
                       "apply_us": wm["kms"] * 1e3, "metadata_us": wm["meta_ms"] * 1e3,
                       "apply_gbs": wkb / (wm["kms"] * 1e-3) / 1e9,
                       "frac": wkb / (wm["kms"] * 1e-3) / 1e9 / peak,
                       "algorithmic_bytes_per_apply": wkb, "tokens_per_step": wc.T,
                       "launches_per_step": wm["launches_per_step"], "copies": wm["n_rot"],
                       "kernel": apply_kernels(wn, args.kernel_policy, wm["fused"])}
                if not args.no_cpu_baseline:
                    ent["cpu_baseline"] = time_oracle(wn, wc, min_seconds=args.cpu_seconds)
                per[wn] = ent

    ms, e2e_ms, kms, meta_ms = max_over_ranks([ms, e2e_ms, kms, meta_ms], world, dev)
    if rank != 0:
        return 0

    tokens = c.T
    value = whole_job_throughput(tokens, args.steps, world, ms)
    e2e = whole_job_throughput(tokens, e2e_n, world, e2e_ms)
    kbytes = kernel_bytes(name, ab, m["fused"])
    achieved = kbytes / (kms * 1e-3) / 1e9
    n_rot = m["n_rot"]
    line = {
        "metric": "LoRA-delta tokens/s", "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{name}: {WORKLOADS[name]}", "tokens_per_step": tokens,
                   "active_rows": ab["active"],
                   "algorithmic_bytes_per_step": ab["total"],
                   "hbm_gbs_per_step": ab["total"] / (ms / args.steps * 1e-3) / 1e9,
                   "l2": f"inputs rotate over {n_rot} resident copies "
                         f"({n_rot * ab['total'] / 1e6:.0f} MB of algorithmic bytes, L2 {l2 / 1e6:.0f} MB)",
                   "timing": f"one CUDA graph of exactly {args.steps} steps (metadata + apply each, one lora_build_meta_apply call for a dense layer; rotating "
                             f"copies), replayed once untimed and once between CUDA events",
                   "parallelism": f"replicas{world}",
                   "metadata_us_alone": meta_ms * 1e3, "apply_us_alone": kms * 1e3,
                   "per_workload": per},
        "roofline": {"bound": "hbm", "kernel": apply_kernels(name, args.kernel_policy, m["fused"]),
                     "achieved": achieved, "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic(name, "moe" if moe else "apply"),
                     "algorithmic_bytes_per_launch": kbytes, "avg_launch_us": kms * 1e3},
        "clocks": cs.summary(),
        "e2e": {"value": e2e, "unit": "tokens/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                "steps": e2e_n,
                "timing": (f"CUDA graphs of {G} steps pipelined over {NSET} buffer sets: pinned H2D copies "
                           "(copy stream), metadata + apply (compute stream), D2H copy (second copy stream)")
                          if e2e_graph is not None else "eager pipelined calls"},
        "gpu_launches": m["launches_per_step"] * args.steps,
    }
    if name == "linear_prefill":
        # a dense contraction: the roofline is the tensor pipe's
        tpk, tkind = load_tensor_peak()
        fl = linear_flops(c)
        line["roofline"] = {"bound": "tensor", "kernel": apply_kernels(name, args.kernel_policy, m["fused"]),
                            "achieved": fl / (kms * 1e-3) / 1e12, "peak": tpk,
                            "peak_kind": f"{tkind} bf16_tflops_sustained", "unit": "TFLOP/s",
                            "frac": fl / (kms * 1e-3) / 1e12 / tpk, "traffic": None,
                            "algorithmic_flops_per_launch": fl, "avg_launch_us": kms * 1e3}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = time_oracle(name, c, min_seconds=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="decode_qkv", choices=sorted(WORKLOADS))
    ap.add_argument("--max-copies", type=int, default=16)
    ap.add_argument("--kernel-launches", type=int, default=200)
    ap.add_argument("--clock-seconds", type=float, default=1.0)
    ap.add_argument("--cpu-seconds", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only --workload (skip the per_workload block of the other configurations)")
    ap.add_argument("--kernel-policy", type=int, default=0, choices=[0, 1, 2, 3, 4, 5, 6, 7, 8],
                    help="lora_set_kernel_policy: 0 automatic, 1 persistent split-K kernel, 2 cluster kernel "
                         "first, 3 no fused decode / MoE block kernel, 4 MoE per-pair blocks, 5 MoE block kernel "
                         "over the metadata's tiles, 6 the linear layer as one tcgen05 GEMM with the delta in its "
                         "accumulator, 7 fused decode kernel up to 32 rows per slot, 8 split expand on warp-level MMAs (tuning)")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        return run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

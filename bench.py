#!/usr/bin/env python
"""Decode throughput of the batch-invariant forward on GB300.

One step = one greedy decode step of a Qwen3-8B-shaped random-init model (36
layers, d 4096, 32/8 heads, head_dim 128, FFN 12288, vocab 151936) for a batch
of 64 requests whose cached KV lengths are drawn uniform on [128, 4096]:
embedding, per layer RMSNorm -> QKV GEMM -> q/k head RMSNorm + RoPE + paged KV
store -> split-KV attention + merge tree -> O GEMM (+residual) -> RMSNorm ->
gate|up GEMM with SwiGLU in its epilogue -> down GEMM (+residual), then final RMSNorm, lm-head
(fp32 logits) and top-20.  All of it runs in libbi's kernels through bi_model_forward; timed steps replay
a CUDA graph captured from one bi_model_forward call (the step's positions and ids staged into its fixed
buffers), the per-kernel profile pass calls it eagerly.

Prints one JSON line (rank 0).  --impl reference times the float64 CPU oracle
on a bounded sample of the same workload instead.
Multi-GPU: replicas only (every rank decodes its own batch; no collective on
the data path); value = tokens of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "invariant decode tok/s (8B-shape, B=1..64); GEMM TFLOP/s & attn GB/s vs peak"
BATCH = 64
KV_LO, KV_HI = 128, 4096
TOPK = 20
SWEEP_BATCHES = (1, 8)
GEMM_SWEEP_M = (256, 1024, 4096)
GEMM_SWEEP_N = (4096, 14336, 151936)
GEMM_SWEEP_K = 4096
WORKLOAD = ("Qwen3-8B-shaped decode step (36 layers, d4096, 32/8 heads, hd128, q/k head RMSNorm, FFN 12288, vocab 151936), "
            "B=64 requests, cached KV lengths U{128..4096}, greedy top-20")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--mode", choices=["invariant", "fast", "protected", "invariant_ksplit"], default="invariant")
    ap.add_argument("--batch", type=int, default=BATCH)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None, help="keep the raw SM clock samples of the timed region here")
    ap.add_argument("--case", choices=["model", "attn", "gemm", "gemm_swiglu", "topk", "rmsnorm"], default="model",
                    help="model: the decode-step workload; attn/gemm/gemm_swiglu/topk/rmsnorm: one kernel on a "
                         "small case (for profiler captures), printing that kernel's timing")
    ap.add_argument("--gemm-shape", default="64,24576,4096",
                    help="M,N,K of --case gemm (gemm_swiglu: N = 2F, the gate and up rows)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the GEMM sweep, RMSNorm roofline and smaller decode batches")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


# ---------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, path: str | None = None):
        """path: where the raw nvidia-smi samples go (a temporary file when not given)."""
        self.proc = None
        self.tmp = path is None
        if path is None:
            import tempfile
            fd, path = tempfile.mkstemp(prefix="bi_clocks_", suffix=".csv")
            os.close(fd)
        self.path = path
        self.gpu = gpu_index

    def start(self):
        try:
            os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            if self.tmp and os.path.exists(self.path):
                os.remove(self.path)
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            lines = f.readlines()
        if self.tmp:
            os.remove(self.path)
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------- replicas (N > 1)
def replica_seeds(seed: int, rank: int) -> dict:
    """Seeds of one rank's replica: its own weights, KV lengths and cached
    histories, so every rank decodes a different batch (no data is shared)."""
    return {"weights": seed + 1000 * rank, "kv_lens": seed + 17 * rank, "history": seed * 7919 + rank}


def max_over_ranks(x: float, dist, device) -> float:
    """The largest of the ranks' values: the job takes as long as its slowest rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(batch: int, world: int, steps: int, seconds: float) -> float:
    """Tokens per second of the whole job: every rank decodes `batch` tokens per step."""
    return batch * world * steps / seconds


# ---------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local_rank):
    import torch

    import synth
    import invariant_deterministic_02_gb300 as bi
    from invariant_deterministic_02_gb300.model import QWEN3_8B, BiModel

    torch.cuda.set_device(local_rank)
    dev = "cuda"
    mode = bi.MODES[args.mode]
    B = args.batch
    K, W = args.steps, args.warmup
    shape = QWEN3_8B
    seeds = replica_seeds(args.seed, rank)
    Ls = synth.uniform_ints(B, KV_LO, KV_HI, seeds["kv_lens"])  # KV length at the first step
    compare = ([m for m in ("fast", "invariant_ksplit", "protected") if m != args.mode]
               if args.mode == "invariant" else [])
    act32 = args.mode == "invariant"  # also time the fp32-activation variant of the same step
    sweep_b = [b for b in SWEEP_BATCHES if b < B] if args.mode == "invariant" and not args.no_extras else []
    tune = "fast" in compare
    # warm-up, timed, profiled, end-to-end, other modes, fp32 activations, smaller decode batches, FAST tuning
    total_steps = (W + 2 * K + K + len(compare) * (K + 1) + (K + 1 if act32 else 0) +
                   len(sweep_b) * (W + K) + (3 * (K + 1) if tune else 0))
    pages = int(sum((int(L) + total_steps + 16) // 16 + 1 for L in Ls)) + 16
    model = BiModel(shape, BiModel.random_weights(shape, seed=seeds["weights"]), num_pages=pages,
                    page_seed=args.seed + 3)
    for b in range(B):
        model.install_history(b, int(Ls[b]) - 1, seeds["history"] + 131 * b)
    # block table covering every step; pos0 of step s is L_b - 1 + s
    rows = [model.pool.ensure(b, int(Ls[b]) + total_steps) for b in range(B)]
    max_pages = max(len(r) for r in rows)
    bt = np.full((B, max_pages), -1, dtype=np.int32)
    for b, r in enumerate(rows):
        bt[b, :len(r)] = r
    pos_all = (Ls[None, :].astype(np.int64) - 1 + np.arange(total_steps)[:, None]).astype(np.int32)
    d_bt = torch.from_numpy(bt).to(dev)
    d_qs = torch.arange(B + 1, dtype=torch.int32, device=dev)
    d_pos = torch.from_numpy(pos_all).to(dev)
    ids = [torch.from_numpy(synth.token_ids(B, shape.vocab, args.seed + 5)).to(dev),
           torch.empty(B, dtype=torch.int32, device=dev)]
    logits = torch.empty((B, shape.vocab), dtype=torch.float32, device=dev)
    tv = torch.empty((B, TOPK), dtype=torch.float32, device=dev)
    ti = torch.empty((B, TOPK), dtype=torch.int32, device=dev)
    target = 0 if args.mode == "protected" else -1

    def batch_for(step, m=None, nb=B):
        # PROTECTED protects request 0 (its one token row); nb < B: the first nb requests
        t = 0 if (m if m is not None else mode) == bi.PROTECTED else -1
        return bi.Batch(nb, nb, 1, d_qs.data_ptr(), d_pos[step].data_ptr(), d_bt.data_ptr(), max_pages, pages,
                        t, 0 if t >= 0 else -1, 1 if t >= 0 else 0)

    dims32 = bi.ModelDims.from_buffer_copy(model.dims)  # same model, fp32 activations
    dims32.act_f32 = 1
    ws_bytes = max(bi.bi_model_workspace(model.dims, batch_for(0, bi.MODES[m]), bi.MODES[m])
                   for m in [args.mode] + compare)
    if act32:
        ws_bytes = max(ws_bytes, bi.bi_model_workspace(dims32, batch_for(0), mode))
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sp = stream.cuda_stream
    step = [0]

    # Timed decode steps replay a CUDA graph of bi_model_forward, captured once per (mode, activations, batch
    # size) on fixed buffers: the step's positions are copied into a fixed buffer before the replay and its
    # greedy ids fed back after it (two small device copies).  The profiled pass runs the same steps eagerly.
    d_pos1 = d_pos[0].clone()
    d_in = ids[0].clone()
    d_next = torch.empty(B, dtype=torch.int32, device=dev)
    graphs = {}

    def graph_for(m, dims, nb):
        key = (m, int(dims.act_f32), nb)
        if key not in graphs:
            t = 0 if m == bi.PROTECTED else -1
            bat = bi.Batch(nb, nb, 1, d_qs.data_ptr(), d_pos1.data_ptr(), d_bt.data_ptr(), max_pages, pages,
                           t, 0 if t >= 0 else -1, 1 if t >= 0 else 0)

            def call(st, bat=bat, m=m, dims=dims):
                bi.bi_model_forward(dims, model.mw, model.rope_cos, model.rope_sin, d_in, bat, model.k_ptrs,
                                    model.v_ptrs, logits, TOPK, tv, ti, greedy_ids=d_next, mode=m, workspace=ws,
                                    ws_bytes=ws_bytes, stream=st)
            graphs[key] = (StepGraph(torch, call), bat)
        return graphs[key][0]

    def one_step(m=mode, dims=model.dims, nb=B, eager=False):
        s = step[0]
        if eager:
            src, dst = ids[s % 2], ids[(s + 1) % 2]
            bi.bi_model_forward(dims, model.mw, model.rope_cos, model.rope_sin, src, batch_for(s, m, nb),
                                model.k_ptrs, model.v_ptrs, logits, TOPK, tv, ti, greedy_ids=dst, mode=m,
                                workspace=ws, ws_bytes=ws_bytes, stream=sp)
        else:
            d_pos1.copy_(d_pos[s])
            g = graph_for(m, dims, nb)
            g.replay()
            d_in.copy_(d_next)
        step[0] += 1

    dist = None
    if world > 1:
        import torch.distributed as dist
    for _ in range(W):
        one_step()
    torch.cuda.synchronize()

    # ---------------------------------------------------------------- timed region (device-resident inputs)
    clocks = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else
                          int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank]),
                          args.clocks_csv if world == 1 else None)
    clocks.start()
    time.sleep(0.3)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(K):
        one_step()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    ck = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    ms_per_step = ms / K
    value = job_throughput(B, world, K, ms / 1000.0)
    assert bi.bi_device_error() == 0

    # ---------------------------------------------------------------- profiled pass: per-kernel event timing
    bi.bi_profile_start(K * 600)
    p_step0 = step[0]
    for _ in range(K):
        one_step(eager=True)
    torch.cuda.synchronize()
    bi.bi_profile_stop()
    kern = {}
    tot_ms = 0.0
    for name in bi.bi_profile_kernels():
        n, t = bi.bi_profile_read(name)
        if n:
            kern[name] = {"launches_per_step": n / K, "ms_per_step": t / K}
            tot_ms += t / K
    for v in kern.values():
        v["share"] = v["ms_per_step"] / tot_ms if tot_ms > 0 else None
    launches_per_step = sum(v["launches_per_step"] for v in kern.values())
    # algorithmic bytes / flops of the profiled steps
    L = shape.layer
    kvlens = pos_all[p_step0:p_step0 + K] + 1  # [K][B]
    kv_bytes_step = float(kvlens.sum(axis=1).mean()) * L.n_kv_heads * L.head_dim * 2 * 2 * shape.n_layers
    q_bytes_step = B * L.n_q_heads * L.head_dim * 2 * shape.n_layers
    gemm_shapes = [(L.qkv_dim, L.d_model), (L.d_model, L.n_q_heads * L.head_dim), (2 * L.ffn_dim, L.d_model),
                   (L.d_model, L.ffn_dim)]
    gemm_bytes_step, gemm_flops_step = 0.0, 0.0
    # with no SwiGLU launch the gate|up GEMM applied it in its epilogue and wrote only the [B][F] activation
    swiglu_fused = "swiglu" not in kern
    for N, Kd in gemm_shapes:
        n_out = N // 2 if (swiglu_fused and N == 2 * L.ffn_dim) else N
        gemm_bytes_step += shape.n_layers * (2 * (B * Kd + N * Kd) + 2 * B * n_out +
                                             (2 * B * N if N == L.d_model else 0))
        gemm_flops_step += shape.n_layers * 2.0 * B * N * Kd
    gemm_bytes_step += 2 * (B * L.d_model + shape.vocab * L.d_model) + 4 * B * shape.vocab
    gemm_flops_step += 2.0 * B * shape.vocab * L.d_model
    pk = peaks()
    algo = {"attn_decode_split": (kv_bytes_step + q_bytes_step, "hbm"), "gemm": (gemm_bytes_step, "hbm")}
    dom = max(kern.items(), key=lambda kv: kv[1]["ms_per_step"])[0]
    roof_name = dom if dom in algo else max(algo, key=lambda n: kern.get(n, {}).get("ms_per_step", 0))
    kb, bound = algo[roof_name]
    kms = kern[roof_name]["ms_per_step"]
    achieved = kb / (kms / 1000.0) / 1e9
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if os.path.exists(tpath):
        tj = json.load(open(tpath))
        ent = tj.get(roof_name)
        if ent and ent.get("source_sha") == _source_sha(ent.get("source")):
            traffic = ent.get("bytes_per_launch")
    launches_roof = kern[roof_name]["launches_per_step"]
    roofline = {"kernel": roof_name, "bound": bound, "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                "traffic": traffic, "algorithmic_bytes_per_launch": round(kb / launches_roof),
                "launch_ms": round(kms / launches_roof, 5), "peak_src": pk["src"] + " hbm_gbs (STREAM-style copy)"}
    others = {}
    for n, (b_, _) in algo.items():
        if n in kern and n != roof_name:
            a = b_ / (kern[n]["ms_per_step"] / 1000.0) / 1e9
            others[n] = {"achieved_GBs": round(a, 1), "frac_hbm": round(a / pk["hbm_gbs"], 4)}
    if "gemm" in kern:
        others.setdefault("gemm", {})["achieved_TFLOPs"] = round(gemm_flops_step / (kern["gemm"]["ms_per_step"] /
                                                                                    1000.0) / 1e12, 2)

    # ---------------------------------------------------------------- end to end through host buffers
    # The step's inputs (token ids, positions, the batch's row starts and block table) travel in one pinned
    # host buffer and one copy to one device buffer that the batch descriptor points into; the step's top-20
    # values and ids come back in one copy; the next step's ids are the top-1 of this one.
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_pos_all = pin(pos_all)
    al = lambda n: (n + 3) // 4 * 4  # int32 offsets kept 16-byte aligned
    o_ids, o_pos, o_qs = 0, al(B), 2 * al(B)
    o_bt = o_qs + al(B + 1)
    n_in = o_bt + bt.size
    h_in = torch.empty(n_in, dtype=torch.int32).pin_memory()
    h_in[o_ids:o_ids + B] = torch.from_numpy(synth.token_ids(B, shape.vocab, args.seed + 6))
    h_in[o_qs:o_qs + B + 1] = torch.arange(B + 1, dtype=torch.int32)
    h_in[o_bt:o_bt + bt.size] = torch.from_numpy(np.ascontiguousarray(bt).reshape(-1))
    h_in[o_pos:o_pos + B] = h_pos_all[step[0]]
    d_in_e = h_in.to(dev)
    out_e = torch.empty(2 * B * TOPK, dtype=torch.int32, device=dev)  # [top-20 values as fp32 bits | top-20 ids]
    tv_e = out_e[:B * TOPK].view(torch.float32).view(B, TOPK)
    ti_e = out_e[B * TOPK:].view(B, TOPK)
    h_out = torch.empty(2 * B * TOPK, dtype=torch.int32).pin_memory()
    h_out_i = h_out[B * TOPK:].view(B, TOPK)
    base = d_in_e.data_ptr()
    b_e = bi.Batch(B, B, 1, base + 4 * o_qs, base + 4 * o_pos, base + 4 * o_bt, max_pages, pages, target,
                   0 if target >= 0 else -1, 1 if target >= 0 else 0)
    d_ids = d_in_e[o_ids:o_ids + B]

    def e2e_step(st):
        # one graph per step: the copy of the step's inputs from pinned host memory, the public call, and the
        # copy of its top-20 back (both copies are graph nodes that read / write the pinned buffers at replay)
        d_in_e.copy_(h_in, non_blocking=True)
        bi.bi_model_forward(model.dims, model.mw, model.rope_cos, model.rope_sin, d_ids, b_e, model.k_ptrs,
                            model.v_ptrs, logits, TOPK, tv_e, ti_e, greedy_ids=None, mode=mode, workspace=ws,
                            ws_bytes=ws_bytes, stream=st)
        h_out.copy_(out_e, non_blocking=True)

    g_e = StepGraph(torch, e2e_step)
    h2d = 4 * n_in
    d2h = 4 * 2 * B * TOPK
    # host-side updates through numpy views of the pinned buffers (no torch dispatch on the host path)
    h_in_np, h_ids_np, h_pos_np = h_in.numpy(), h_out_i.numpy(), h_pos_all.numpy()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(K):
        h_in_np[o_pos:o_pos + B] = h_pos_np[step[0]]
        g_e.replay()
        stream.synchronize()
        h_in_np[o_ids:o_ids + B] = h_ids_np[:, 0]
        step[0] += 1
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)
    e2e = {"value": round(job_throughput(B, world, K, e2e_s), 2), "unit": "tok/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h}

    # ---------------------------------------------------------------- the same steps in the other modes
    # FAST: the non-invariant schedule (cost of invariance = FAST / INVARIANT throughput);
    # INVARIANT_KSPLIT: the K-only split-K GEMM variant (also batch invariant);
    # invariant_act_f32: INVARIANT with fp32 activations (bf16 weights and KV cache)
    modes = {}
    runs = [(m, bi.MODES[m], model.dims) for m in compare] + ([("invariant_act_f32", mode, dims32)] if act32 else [])
    for name, m, dims in runs:
        one_step(m, dims)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(K):
            one_step(m, dims)
        c1.record(stream)
        torch.cuda.synchronize()
        cms = c0.elapsed_time(c1)
        cms = max_over_ranks(cms, dist, dev)
        modes[name] = {"value": round(job_throughput(B, world, K, cms / 1000.0), 2), "unit": "tok/s",
                       "ms_per_step": round(cms / K, 4)}
    if "fast" in modes:
        modes["invariant_over_fast_time"] = round(ms_per_step / modes["fast"]["ms_per_step"], 4)
    if "protected" in modes:
        modes["protected"]["target_request"] = 0

    # ---------------------------------------------------------------- FAST tuned by timing
    # The non-invariant schedule at its best: every GEMM shape of the step takes whichever of FAST's
    # split-K rule and INVARIANT's tile plan times faster here, and decode attention whichever of the
    # occupancy-chosen split count and the 256-token splits gives the faster FAST step.
    if tune:
        L = shape.layer
        shapes_nk = [(L.qkv_dim, L.d_model), (L.d_model, L.n_q_heads * L.head_dim), (2 * L.ffn_dim, L.d_model),
                     (L.d_model, L.ffn_dim), (shape.vocab, L.d_model)]
        flush = L2Flush(torch)
        gemm_choice = {}
        for N, Kd in shapes_nk:
            A = synth.normal_device((B, Kd), 700 + N)
            Wt = synth.normal_device((N, Kd), 701 + N, std=0.02)
            C = torch.empty((B, N), dtype=torch.float32 if N == shape.vocab else torch.bfloat16, device=dev)
            gws = torch.empty(max(1, bi.lib().bi_gemm_workspace(B, N, Kd, bi.FAST)), dtype=torch.uint8, device=dev)
            t = {}
            for plan in (0, 1):
                bi.bi_fast_gemm_plan(B, N, Kd, plan)
                f = lambda: bi.bi_gemm(A, Wt, C, mode=bi.FAST, workspace=gws)
                for _ in range(3):
                    f()
                t[plan] = time_launches(torch, f, 10, flush)
            best = min(t, key=t.get)
            bi.bi_fast_gemm_plan(B, N, Kd, best)
            graphs.clear()  # captured FAST steps carry the plans they were captured with
            gemm_choice["%dx%dx%d" % (B, N, Kd)] = {"plan": ["split_k", "tile_plan"][best],
                                                   "ms": {"split_k": round(t[0], 4), "tile_plan": round(t[1], 4)}}
            del A, Wt, C, gws
        step_ms = {}
        for plan in (0, 1):
            bi.bi_fast_attention_plan(plan)
            graphs.clear()
            one_step(bi.FAST)
            torch.cuda.synchronize()
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(stream)
            for _ in range(K):
                one_step(bi.FAST)
            c1.record(stream)
            torch.cuda.synchronize()
            step_ms[plan] = c0.elapsed_time(c1) / K
        attn_best = min(step_ms, key=step_ms.get)
        bi.bi_fast_attention_plan(attn_best)
        graphs.clear()
        one_step(bi.FAST)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(K):
            one_step(bi.FAST)
        c1.record(stream)
        torch.cuda.synchronize()
        cms = max_over_ranks(c0.elapsed_time(c1), dist, dev)
        modes["fast_tuned"] = {"value": round(job_throughput(B, world, K, cms / 1000.0), 2), "unit": "tok/s",
                               "ms_per_step": round(cms / K, 4), "gemm_plans": gemm_choice,
                               "attention_plan": ["occupancy_split_count", "splits_of_256"][attn_best],
                               "attention_step_ms": {"occupancy_split_count": round(step_ms[0], 4),
                                                     "splits_of_256": round(step_ms[1], 4)}}
        modes["invariant_over_fast_tuned_time"] = round(ms_per_step / modes["fast_tuned"]["ms_per_step"], 4)
        # back to FAST's own rules
        bi.bi_fast_attention_plan(0)
        for N, Kd in shapes_nk:
            bi.bi_fast_gemm_plan(B, N, Kd, 0)
        graphs.clear()

    # ---------------------------------------------------------------- smaller decode batches (B = 1, 8)
    # the first nb requests of the same model and caches; roofline: the weights every step streams
    # (all layers + lm-head) plus the KV of those requests, against the measured HBM copy bandwidth
    w_bytes = weight_bytes_per_step(shape)
    decode_sweep = {}
    for nb in sweep_b:
        for _ in range(W):
            one_step(mode, model.dims, nb)
        torch.cuda.synchronize()
        s0 = step[0]
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(K):
            one_step(mode, model.dims, nb)
        c1.record(stream)
        torch.cuda.synchronize()
        cms = max_over_ranks(c0.elapsed_time(c1), dist, dev) / K
        kvb = float((pos_all[s0:s0 + K, :nb] + 1).sum(axis=1).mean()) * L.n_kv_heads * L.head_dim * 4 * shape.n_layers
        gbs = (w_bytes + kvb) / (cms / 1000.0) / 1e9
        decode_sweep["B%d" % nb] = {"value": round(nb * world / (cms / 1000.0), 2), "unit": "tok/s",
                                    "ms_per_step": round(cms, 4), "bytes_per_step": round(w_bytes + kvb),
                                    "achieved_GBs": round(gbs, 1), "frac_hbm": round(gbs / pk["hbm_gbs"], 4)}
    kvb64 = kv_bytes_step
    gbs64 = (w_bytes + kvb64) / (ms_per_step / 1000.0) / 1e9
    decode_sweep["B%d" % B] = {"value": round(value, 2), "unit": "tok/s", "ms_per_step": round(ms_per_step, 4),
                               "bytes_per_step": round(w_bytes + kvb64), "achieved_GBs": round(gbs64, 1),
                               "frac_hbm": round(gbs64 / pk["hbm_gbs"], 4), "note": "the headline run"}
    assert bi.bi_device_error() == 0

    line = {"metric": METRIC, "value": round(value, 2), "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic: seeded random-init weights ~N(0,0.02), random token ids, "
                                     "seeded N(0,1) KV history",
            "config": {"workload": WORKLOAD, "batch_per_gpu": B, "kv_len": "U{%d..%d} seed %d" % (KV_LO, KV_HI,
                                                                                            args.seed),
                       "mode": args.mode, "parallelism": "replicas" if world > 1 else "single",
                       "launch": "each step replays a CUDA graph of one bi_model_forward call (stream capture of "
                                 "the public call, same kernels); the per-kernel profile runs the steps eagerly",
                       "l2": "inputs larger than L2: ~15 GB weights + ~20 GB KV streamed per step"},
            "clocks": ck, "e2e": e2e, "gpu_launches": int(round(launches_per_step * K)),
            "roofline": roofline, "kernels": {k: {kk: (round(vv, 5) if isinstance(vv, float) else vv)
                                                  for kk, vv in v.items()} for k, v in kern.items()},
            "other_rooflines": others, "modes": modes}
    if decode_sweep:
        line["decode_batch_sweep"] = decode_sweep
    return line


def _source_sha(rel):
    import hashlib
    if not rel:
        return None
    p = os.path.join(ROOT, rel)
    if not os.path.exists(p):
        return None
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def weight_bytes_per_step(shape) -> float:
    """Bytes of weights one decode step streams: every layer's projections and
    norms, the final norm and the lm-head (the embedding rows gathered are B rows)."""
    L = shape.layer
    per_layer = (L.qkv_dim * L.d_model + L.d_model * L.n_q_heads * L.head_dim + 2 * L.ffn_dim * L.d_model +
                 L.d_model * L.ffn_dim + 2 * L.d_model + (2 * L.head_dim if L.qk_norm else 0))
    return 2.0 * (shape.n_layers * per_layer + L.d_model + shape.vocab * L.d_model)


class StepGraph:
    """One call of the public bi_model_forward captured in a CUDA graph (stream capture) on fixed buffers and
    replayed on the current stream: the same kernels with the same arguments, launched as one graph.  The call
    runs once eagerly on the capture stream first (lazy initialisation happens outside the capture)."""

    def __init__(self, torch, call):
        cur = torch.cuda.current_stream()
        side = torch.cuda.Stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            call(side.cuda_stream)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            call(torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()

    def replay(self):
        self.graph.replay()


class L2Flush:
    """Writes a buffer larger than L2 (129 MB) between timed launches, then reads a second one of the same
    size: the write evicts whatever the previous launch left in L2, and the read evicts the write's own dirty
    lines, so the timed launch starts with an L2 that holds none of its inputs and owes DRAM no write-backs
    of the flush."""

    def __init__(self, torch):
        self.torch = torch
        self.buf = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
        self.rbuf = torch.ones(64 * 1024 * 1024, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.buf.fill_(1)
        self.torch.sum(self.rbuf)


def busy(torch):
    """Keeps the GPU busy for ~0.1 ms (a spin kernel) while the host enqueues the next timed launch, so
    that the launch's start event is not recorded on an idle GPU ahead of the host's launch overhead."""
    torch.cuda._sleep(200000)


def time_launches(torch, fn, reps: int, flush) -> float:
    """Median milliseconds of `fn` over `reps` launches, each bracketed by CUDA events on
    the current (launching) stream, L2 flushed before each."""
    st = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        flush()
        busy(torch)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        fn()
        e1.record(st)
        e1.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def gemm_sweep(torch, bi, synth, pk, warmup: int, reps: int) -> dict:
    """INVARIANT bi_gemm over the GEMM-sweep shapes at M >= 256 (K = 4096; bf16 out, fp32 out for the
    lm-head width N = 151936), timed alone with L2 flushed: TFLOP/s against the burst bf16 peak and
    against the roofline min(peak, AI * HBM); cuBLAS (torch.matmul, bf16 out) on the same operands for
    context."""
    flush = L2Flush(torch)
    out = {}
    Kd = GEMM_SWEEP_K
    peak_t = pk["bf16_tflops"]
    for N in GEMM_SWEEP_N:
        W = synth.normal_device((N, Kd), 900 + N, std=0.02)
        for M in GEMM_SWEEP_M:
            A = synth.normal_device((M, Kd), 800 + M)
            f32 = N == 151936
            C = torch.empty((M, N), dtype=torch.float32 if f32 else torch.bfloat16, device="cuda")
            fn = lambda: bi.bi_gemm(A, W, C)
            for _ in range(warmup):
                fn()
            ms = time_launches(torch, fn, reps, flush)
            flops = 2.0 * M * N * Kd
            byts = 2.0 * (M * Kd + N * Kd) + (4 if f32 else 2) * M * N
            tf = flops / (ms / 1000.0) / 1e12
            roof = min(peak_t, flops / byts * pk["hbm_gbs"] * 1e9 / 1e12)
            cb = lambda: torch.matmul(A, W.t())
            for _ in range(2):
                cb()
            cms = time_launches(torch, cb, reps, flush)
            out["M%d_N%d" % (M, N)] = {"ms": round(ms, 4), "TFLOPs": round(tf, 1), "frac_peak": round(tf / peak_t, 4),
                                       "roofline_TFLOPs": round(roof, 1), "frac_roofline": round(tf / roof, 4),
                                       "out": "f32" if f32 else "bf16",
                                       "cublas_TFLOPs": round(flops / (cms / 1000.0) / 1e12, 1)}
            del A, C
        del W
    torch.cuda.synchronize()
    return {"K": Kd, "peak_TFLOPs": peak_t, "peak_src": pk["src"] + " bf16_tflops (burst, kernel timed alone)",
            "l2": "flushed before each launch (256 MB written, then another 256 MB read: no dirty lines left)", "shapes": out}


def rmsnorm_roofline(torch, bi, synth, pk, warmup: int, reps: int) -> dict:
    """INVARIANT bi_rmsnorm on 16384 rows x 4096 bf16 (one CTA per row): GB/s of the algorithmic bytes
    (each row read once and written once, gamma once) against the measured HBM copy bandwidth."""
    rows, d = 16384, 4096
    x = synth.normal_device((rows, d), 501)
    g = synth.normal_device((d,), 502, std=0.1, mean=1.0)
    y = torch.empty_like(x)
    fn = lambda: bi.bi_rmsnorm(x, g, y, 1e-5)
    for _ in range(warmup):
        fn()
    ms = time_launches(torch, fn, reps, L2Flush(torch))
    byts = 2.0 * rows * d * 2 + 2 * d
    gbs = byts / (ms / 1000.0) / 1e9
    return {"rows": rows, "d": d, "dtype": "bf16", "ms": round(ms, 4), "achieved_GBs": round(gbs, 1),
            "peak": pk["hbm_gbs"], "frac": round(gbs / pk["hbm_gbs"], 4), "bytes_per_launch": byts}


# ---------------------------------------------------------------------------- oracle (CPU) arm
class OracleSample:
    """A bounded sample of the bench workload for the float64 CPU oracle.

    One decode step of the same 64-request batch (same KV-length draw, seeded
    weights and N(0,1) KV history) through one Qwen3-8B-shaped layer, plus the
    lm-head and top-20 over a 1/16 slice of the vocabulary; the time is scaled
    to 36 layers and the full vocabulary.
    """

    def __init__(self, args):
        import oracle
        import synth

        self.oracle = oracle
        self.shape = synth.QWEN3_8B_LAYER
        self.B = args.batch
        sh = self.shape
        self.Ls = synth.uniform_ints(self.B, KV_LO, KV_HI, args.seed)
        self.w = {k: v.double().numpy() for k, v in synth.layer_weights(sh, args.seed + 77).items()}
        self.h = synth.normal((self.B, sh.d_model), args.seed + 78).double().numpy()
        rng = np.random.default_rng(args.seed + 79)
        self.hist = [(rng.standard_normal((int(L) - 1, sh.n_kv_heads, sh.head_dim)),
                      rng.standard_normal((int(L) - 1, sh.n_kv_heads, sh.head_dim))) for L in self.Ls]
        self.head = synth.normal((151936 // 16, sh.d_model), args.seed + 80, std=0.02).double().numpy()
        self.text = ("one decode step of the %d-request batch through 1 of 36 Qwen3-8B-shaped layers plus "
                     "lm-head/top-20 over 1/16 of the vocabulary (float64 numpy), time scaled x36 layers and "
                     "x16 vocabulary" % self.B)

    def step_seconds(self):
        """Scaled seconds of one full decode step, and the CPU seconds actually spent."""
        o, sh = self.oracle, self.shape
        kv = o.OracleKV(1, sh.n_kv_heads, sh.head_dim)
        for b, (K, V) in enumerate(self.hist):
            kv.set(0, b, K, V)
        a = time.perf_counter()
        o.layer_forward(self.h, self.w, sh, kv, 0, [(b, 1) for b in range(self.B)], [int(L) - 1 for L in self.Ls])
        t_layer = time.perf_counter() - a
        a = time.perf_counter()
        x = o.round_bf16(o.rmsnorm(self.h, np.ones(sh.d_model), sh.rms_eps))
        o.topk(o.round_f32(o.gemm(x, self.head)), TOPK)
        t_head = time.perf_counter() - a
        return 36 * t_layer + 16 * t_head, t_layer + t_head


def run_reference(args):
    cores = len(os.sched_getaffinity(0))
    smp = OracleSample(args)
    for _ in range(max(0, args.warmup)):
        smp.step_seconds()
    scaled, spent = [], 0.0
    for _ in range(args.steps):
        t, c = smp.step_seconds()
        scaled.append(t)
        spent += c
    value = args.batch / statistics.mean(scaled)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1000 * statistics.mean(scaled), 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic: seeded weights ~N(0,0.02), seeded N(0,1) KV history",
            "config": {"workload": WORKLOAD, "batch_per_gpu": args.batch, "kv_len": "U{%d..%d} seed %d" % (
                KV_LO, KV_HI, args.seed), "mode": "oracle (float64 definitions)"},
            "cpu_baseline": {"value": round(value, 4), "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": smp.text + "; %.1f s of CPU work over %d steps" % (spent, args.steps)},
            "e2e": {"value": round(value, 4), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return line


def run_case(args):
    """One kernel on a small case: decode attention over one layer's paged cache
    (B requests, KV U{128..4096}), one GEMM, RMSNorm or top-k over B lm-head rows.  Each launch is
    event-timed on its own (the library's launch timer); cases whose inputs fit in L2 flush it first."""
    import torch

    import synth
    import invariant_deterministic_02_gb300 as bi

    dev = "cuda"
    mode = bi.MODES[args.mode]
    B = args.batch
    K, W = args.steps, args.warmup
    pk = peaks()
    if args.case == "attn":
        hq, hkv, hd = 32, 8, 128
        Ls = synth.uniform_ints(B, KV_LO, KV_HI, args.seed)
        lay = synth.paged_layout(Ls, 16, args.seed + 1)
        kc = synth.normal_device((lay.num_pages, hkv, 16, hd), args.seed + 2)
        vc = synth.normal_device((lay.num_pages, hkv, 16, hd), args.seed + 3)
        q = synth.normal_device((B, hq, hd), args.seed + 4)
        bt = torch.from_numpy(lay.block_table).to(dev)
        kl = torch.from_numpy(Ls).to(dev)
        dims = bi.attn_dims(hq, hkv, hd, lay.max_pages, lay.num_pages)
        out = torch.empty_like(q)
        ws = torch.empty(bi.lib().bi_decode_attention_workspace(B, ctypes.byref(dims), mode), dtype=torch.uint8,
                         device=dev)
        fn = lambda: bi.bi_decode_attention(q, kc, vc, bt, kl, dims, out, mode=mode, workspace=ws)
        kernel, work, unit = "attn_decode_split", float(Ls.sum()) * hkv * hd * 2 * 2 + 2 * B * hq * hd * 2, "GB/s"
        peak = pk["hbm_gbs"]
    elif args.case in ("gemm", "gemm_swiglu"):
        M, N, Kd = (int(v) for v in args.gemm_shape.split(","))
        A = synth.normal_device((M, Kd), args.seed + 5)
        Wt = synth.normal_device((N, Kd), args.seed + 6, std=0.02)
        if args.case == "gemm":
            C = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            fn = lambda: bi.bi_gemm(A, Wt, C, mode=mode)
            n_out = N
        else:
            # the one-call form: the SwiGLU output [M][N/2] is all that is written
            act = torch.empty((M, N // 2), dtype=torch.bfloat16, device=dev)
            ws = torch.empty(max(1, bi.lib().bi_gemm_swiglu_workspace(M, N // 2, Kd, mode)), dtype=torch.uint8,
                             device=dev)
            fn = lambda: bi.bi_gemm_swiglu(A, Wt, act, mode=mode, workspace=ws)
            n_out = N // 2
        flops = 2.0 * M * N * Kd
        byts = 2.0 * (M * Kd + N * Kd + M * n_out)
        if flops / byts > pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9):
            kernel, work, unit, peak = "gemm", flops, "TFLOP/s", pk["bf16_tflops"]
        else:
            kernel, work, unit, peak = "gemm", byts, "GB/s", pk["hbm_gbs"]
    elif args.case == "rmsnorm":
        rows, d = 16384, 4096
        x = synth.normal_device((rows, d), args.seed + 8)
        g = synth.normal_device((d,), args.seed + 9, std=0.1, mean=1.0)
        y = torch.empty_like(x)
        fn = lambda: bi.bi_rmsnorm(x, g, y, 1e-5, mode=mode)
        kernel, work, unit, peak = "rmsnorm", 4.0 * rows * d + 2 * d, "GB/s", pk["hbm_gbs"]
    else:
        V = 151936
        x = synth.normal_device((B, V), args.seed + 7, dtype=torch.float32)
        tv = torch.empty((B, TOPK), dtype=torch.float32, device=dev)
        ti = torch.empty((B, TOPK), dtype=torch.int32, device=dev)
        fn = lambda: bi.bi_topk(x, TOPK, tv, ti)
        kernel, work, unit, peak = "topk", 4.0 * B * V, "GB/s", pk["hbm_gbs"]
    # inputs smaller than L2 (every case but attention) are flushed out of it before each timed launch
    flush = L2Flush(torch) if args.case != "attn" else (lambda: None)
    for _ in range(W):
        fn()
    torch.cuda.synchronize()
    bi.bi_profile_start(K * 8)
    for _ in range(K):
        flush()
        busy(torch)
        fn()
    torch.cuda.synchronize()
    bi.bi_profile_stop()
    n, ms = bi.bi_profile_read(kernel)
    per = ms / n
    achieved = work / (per / 1000.0) / (1e12 if unit == "TFLOP/s" else 1e9)
    return {"case": args.case, "kernel": kernel, "launches": n, "launch_ms": round(per, 5),
            "achieved": round(achieved, 2), "unit": unit, "peak": peak, "frac": round(achieved / peak, 4),
            "work_per_launch": work, "batch": B, "mode": args.mode,
            "shape": args.gemm_shape if args.case in ("gemm", "gemm_swiglu") else None}


def main():
    args = parse()
    if args.case != "model":
        print(json.dumps(run_case(args)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    line = run_ours(args, rank, world, local_rank)
    if args.mode == "invariant" and not args.no_extras:
        import torch

        import synth
        import invariant_deterministic_02_gb300 as bi
        pk = peaks()
        # the memory-bound RMSNorm first: right after the seconds of dense GEMMs of the sweep the part
        # runs at a lower, power-limited clock
        gpu = (local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else
               int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank]))
        for key, run, reps in (("rmsnorm", rmsnorm_roofline, 20), ("gemm_sweep", gemm_sweep, 10)):
            ck = ClockSampler(gpu)
            ck.start()
            time.sleep(0.3)
            line[key] = run(torch, bi, synth, pk, max(3, args.warmup), reps)
            line[key]["clocks"] = ck.stop()
        assert bi.bi_device_error() == 0
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            # sample steps until about 10 s of CPU work (at most 16 steps)
            smp = OracleSample(args)
            runs = []
            while len(runs) < 16 and (len(runs) < 2 or sum(c for _, c in runs) < 10.0):
                runs.append(smp.step_seconds())
            v = args.batch / statistics.mean(t for t, _ in runs)
            line["cpu_baseline"] = {"value": round(v, 4), "unit": "tok/s", "cores": len(os.sched_getaffinity(0)),
                                    "kind": "oracle", "sample": smp.text + "; %d steps, %.1f s of CPU work" %
                                    (len(runs), sum(c for _, c in runs))}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

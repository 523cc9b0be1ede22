"""Benchmark: sparse decode layer-steps/s on the sketch-indexed workload.

Workload (one GPU): 8 requests x 250,000 cached tokens, 16 distinct
full-attention layers, 24 query / 4 KV heads, head dim 256, int8 K/V with a
per-(row, head) fp16 scale, int4 rank-64 key sketch, top-2048 + 64 sinks +
1024-token tail, one pick shared by the 4 KV heads.  Synthetic seeded inputs
(keys with a low-rank dominant subspace), built on the GPU with the library's
own write path.

One step = one decode token for all 8 requests through all 16 layers; per
layer three launches: the appended token's sketch and int8 K/V rows plus the
folded int8 query (a1 + a2, one kernel), the int4 score scan fused with the
radix top-k and the sink/tail union (a3 + a4), and split-K int8 attention
over the resident rows (a5 is the identity, a6).  The 16-layer step is
captured in one CUDA graph.  Layer-steps/s = steps/s x 16; tokens/s = steps/s
x 8.

`--impl reference` times the CPU oracle on the machine's host cores instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse decode layer-steps/s and tokens/s at 8x250K; HBM GB/s vs peak"
UNIT = "layer-steps/s"

W_B, W_T, W_L, W_HQ, W_HKV, W_D, W_R = 8, 250_000, 16, 24, 4, 256, 64
W_K, W_S, W_W = 2048, 64, 1024
MAX_ROWS = W_S + W_K + W_W
SEED = 2
SCAN_BYTES_PER_CAND = W_HKV * W_R // 2          # 128 B sketch row read (keys stay on chip)
ATTN_BYTES_PER_ROW_HEAD = 2 * W_D + 2 * 2       # int8 K + V rows and their fp16 scales

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch from one
# ncu --set full capture of this workload (profiles/ has the summary and the
# command), keyed by a hash of the kernel's sources: a kernel whose sources
# changed since the capture reports null.
MEASURED_TRAFFIC = {
    "score_select": (("common.cuh", "score_common.cuh", "select.cu"), "fd977d44ad3ea622", 258_213_376),
    "attend": (("common.cuh", "attend.cu"), "1f296da7a22ce8c9", 56_068_864),
}


def measured_traffic(kernel):
    import hashlib
    files, digest, nbytes = MEASURED_TRAFFIC[kernel]
    m = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "sparse_kv_long_gb300", "csrc", f), "rb") as fh:
            m.update(fh.read())
    return nbytes if m.hexdigest()[:16] == digest else None


def config_dict(l2_note, layers=W_L):
    return {"workload": f"sketch_8x250000_{layers}L_int4sketch_int8kv", "batch": W_B, "context": W_T,
            "layers": layers, "q_heads": W_HQ, "kv_heads": W_HKV, "head_dim": W_D, "sketch_rank": W_R,
            "top_k": W_K, "sinks": W_S, "tail": W_W, "rows_per_request": MAX_ROWS, "l2": l2_note}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d.get("hbm_gbs", 6800.0)), "measured"
    return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# CPU oracle sample (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------

class OracleSample:
    """One request x one layer of the workload at full context, on the CPU."""

    def __init__(self, seed=SEED):
        import oracle as orc
        import workloads as wl
        self.orc = orc
        orc.build()
        orc.set_threads(os.cpu_count() or 1)
        rng = np.random.default_rng(seed)
        U = wl.orthonormal_basis(W_D, W_R, seed + 1000)
        self.U, self.c = U, wl.sketch_step(W_HKV, W_R, W_D)
        K = wl.to_bf16_bits(wl.lowrank_rows(rng, W_T * W_HKV, U).reshape(W_T, W_HKV, W_D))
        V = wl.to_bf16_bits(rng.standard_normal((W_T, W_HKV, W_D)).astype(np.float32))
        self.q = wl.to_bf16_bits(wl.lowrank_rows(rng, W_HQ, U).reshape(1, W_HQ, W_D))
        self.newk, self.newv = K[-1:].copy(), V[-1:].copy()
        self.sk = orc.sketch_project(K, U, self.c)["q4"].reshape(1, W_T, -1)
        self.k8, self.ks = orc.quant_int8_rows(K)
        self.v8, self.vs = orc.quant_int8_rows(V)
        self.L = np.array([W_T], np.int32)

    def step(self):
        orc = self.orc
        # a1 + row encoding of the appended (current) token
        self.sk[0, -1] = orc.sketch_project(self.newk, self.U, self.c)["q4"][0]
        qk, sk_ = orc.quant_int8_rows(self.newk)
        self.k8[-1], self.ks[-1] = qk[0], sk_[0]
        qv, sv = orc.quant_int8_rows(self.newv)
        self.v8[-1], self.vs[-1] = qv[0], sv[0]
        qq = orc.sketch_query(self.q, W_HKV, self.U, self.c)                     # a2
        sc = orc.index_score(orc.SKETCH_INT4, qq["q8"], self.sk, self.L, S=W_S, W=W_W)  # a3
        idx, cnt = orc.topk_select(sc["okey"], self.L, W_K, S=W_S, W=W_W)          # a4
        return orc.attend(orc.KV_INT8, self.q, self.k8.reshape(W_T, -1), self.v8.reshape(W_T, -1), idx, cnt,
                          1 / math.sqrt(W_D), W_HKV, W_D, W_D, k_scale=self.ks, v_scale=self.vs)  # a6

    def time_steps(self, n=None, budget_s=None):
        times = []
        t_start = time.perf_counter()
        while True:
            t0 = time.perf_counter()
            self.step()
            times.append(time.perf_counter() - t0)
            if n is not None and len(times) >= n:
                break
            if budget_s is not None and time.perf_counter() - t_start >= budget_s:
                break
        return times


def cpu_baseline_block(budget_s=15.0):
    s = OracleSample()
    times = s.time_steps(budget_s=budget_s)
    per_req_layer = statistics.median(times)
    value = 1.0 / (per_req_layer * W_B)  # layer-steps/s (a layer-step covers all 8 requests)
    return {"value": value, "unit": UNIT, "cores": s.orc.max_threads(), "kind": "oracle",
            "sample": f"1 request x 1 layer at 250,000 tokens (a1..a6), {len(times)} runs, median "
                      f"{per_req_layer:.3f} s, scaled x8 requests per layer-step"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    s = OracleSample()
    s.time_steps(n=args.warmup)
    times = s.time_steps(n=args.steps)
    per = float(np.mean(times))
    value = 1.0 / (per * W_B)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * W_B * W_L * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32+f64",
            "data": "synthetic", "config": config_dict("cpu"),
            "cpu_baseline": {"kind": "oracle", "cores": s.orc.max_threads(), "value": value, "unit": UNIT,
                             "sample": "each step: 1 request x 1 layer at 250,000 tokens (a1..a6), "
                                       "scaled x8 requests per layer-step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class ClockSampler:
    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if s[3 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


class SketchWorkloadGPU:
    """Device-resident 16-layer sketch workload and the per-layer step."""

    def __init__(self, torch, skv, wl, device, layers=W_L):
        self.torch, self.skv = torch, skv
        self.L = layers
        dev = device
        gen = wl.device_generator(SEED + 17 * (torch.cuda.current_device() + 1), device=dev)
        U = wl.orthonormal_basis(W_D, W_R, SEED + 1000)
        self.U = torch.from_numpy(U).to(dev)
        self.c = torch.from_numpy(wl.sketch_step(W_HKV, W_R, W_D)).to(dev)
        B, T, L = W_B, W_T, layers
        self.lengths = torch.full((B,), T, dtype=torch.int32, device=dev)
        self.k8 = [torch.empty((B * T, W_HKV, W_D), dtype=torch.int8, device=dev) for _ in range(L)]
        self.v8 = [torch.empty((B * T, W_HKV, W_D), dtype=torch.int8, device=dev) for _ in range(L)]
        self.ks = [torch.empty((B * T, W_HKV), dtype=torch.float16, device=dev) for _ in range(L)]
        self.vs = [torch.empty((B * T, W_HKV), dtype=torch.float16, device=dev) for _ in range(L)]
        self.sk = [torch.empty((B, T, W_HKV * W_R // 2), dtype=torch.uint8, device=dev) for _ in range(L)]
        for l in range(L):
            for b in range(B):
                K = wl.lowrank_rows_torch(gen, T * W_HKV, self.U).view(T, W_HKV, W_D)
                V = wl.randn_torch(gen, (T, W_HKV, W_D), device=dev)
                rows = slice(b * T, (b + 1) * T)
                skv.quantize_int8_rows(K, self.k8[l][rows], self.ks[l][rows])
                skv.quantize_int8_rows(V, self.v8[l][rows], self.vs[l][rows])
                skv.sketch_project(K, self.U, self.c, self.sk[l][b])
                del K, V
        # per-step inputs: query and appended token of every layer
        self.q = wl.lowrank_rows_torch(gen, L * B * W_HQ, self.U).view(L, B, W_HQ, W_D).contiguous()
        self.newk = wl.lowrank_rows_torch(gen, L * B * W_HKV, self.U).view(L, B, W_HKV, W_D).contiguous()
        self.newv = wl.randn_torch(gen, (L, B, W_HKV, W_D), device=dev).contiguous()
        self.new_rows = (torch.arange(B, device=dev, dtype=torch.int64) * T + (T - 1)).contiguous()
        self.q8 = torch.empty((B, W_HKV * W_R), dtype=torch.int8, device=dev)
        self.sigma = torch.empty((B,), dtype=torch.float32, device=dev)
        self.okeys = torch.zeros((B, T), dtype=torch.int32, device=dev)
        self.idx = torch.zeros((B, MAX_ROWS), dtype=torch.int32, device=dev)
        self.cnt = torch.zeros((B,), dtype=torch.int32, device=dev)
        self.tws = torch.zeros((skv.score_select_workspace_size(B),), dtype=torch.uint8, device=dev)
        self.aws = torch.zeros((skv.attend_workspace_size(B, W_HQ, W_HKV, W_D, MAX_ROWS),), dtype=torch.uint8,
                               device=dev)
        self.pws = torch.zeros((skv.decode_prepare_workspace_size(B, W_HKV),), dtype=torch.uint8, device=dev)
        self.out = torch.zeros((L, B, W_HQ, W_D), dtype=torch.float32, device=dev)
        self.status = torch.zeros((1,), dtype=torch.int32, device=dev)
        torch.cuda.synchronize()

    KERNELS_PER_LAYER = 3  # a1 + int8 append + a2 fused, a3 + a4 fused, a6

    def layer(self, l, marks=None):
        skv, st = self.skv, self.status
        ev = (lambda name: marks(l, name)) if marks else (lambda name: None)
        ev("start")
        skv.decode_prepare(self.q[l], self.newk[l], self.newv[l], self.U, self.c, self.new_rows,
                           self.sk[l].view(W_B * W_T, -1), self.k8[l], self.ks[l], self.v8[l], self.vs[l], self.q8,
                           self.pws, sigma=self.sigma)
        ev("scan0")
        skv.score_select(skv.SKETCH_INT4, self.q8, self.sk[l], self.lengths, W_K, self.idx, self.cnt, self.tws,
                         S=W_S, W=W_W, status=st)
        ev("scan1")
        ev("attn0")
        skv.sparse_attend_decode(skv.KV_INT8, self.q[l], self.k8[l], self.v8[l], self.idx, self.cnt,
                                 1 / math.sqrt(W_D), self.out[l], self.aws, W_HKV, k_scale=self.ks[l],
                                 v_scale=self.vs[l], req_row_stride=W_T, status=st)
        ev("attn1")

    def step(self):
        for l in range(self.L):
            self.layer(l)


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import sparse_kv_long_gb300 as skv
    import workloads as wl
    from sparse_kv_long_gb300 import _build

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    _build.build()
    dev = torch.device("cuda", local)

    def barrier():
        if world > 1:
            dist.barrier()

    L = args.layers
    w = SketchWorkloadGPU(torch, skv, wl, dev, layers=L)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    # ---- capture the 16-layer step in one CUDA graph -------------------------------
    with torch.cuda.stream(stream):
        w.step()  # eager warm-up (also sets kernel attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream, capture_error_mode="relaxed"):
        w.step()
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        gpu_id = str(local)
    with ClockSampler(gpu_id) as clk:
        time.sleep(0.3)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            e1.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms_total = e0.elapsed_time(e1)
    if world > 1:
        t = torch.tensor([ms_total], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms_total = float(t.item())
    ms_per_step = ms_total / args.steps
    steps_per_s = 1e3 / ms_per_step
    value = steps_per_s * L * world              # layer-steps/s over all replicas
    tokens_per_s = steps_per_s * W_B * world
    status = int(w.status.item())

    # ---- per-kernel durations: eager launches queued behind a sleep -------------------
    marks = {}

    def mark(l, name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        marks.setdefault(name, []).append(e)

    scan_ms, attn_ms, topk_ms = [], [], []
    for _ in range(3):
        marks.clear()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(50_000_000)
            for l in range(L):
                w.layer(l, mark)
        torch.cuda.synchronize()
        for l in range(L):
            scan_ms.append(marks["scan0"][l].elapsed_time(marks["scan1"][l]))
            topk_ms.append(marks["scan1"][l].elapsed_time(marks["attn0"][l]))
            attn_ms.append(marks["attn0"][l].elapsed_time(marks["attn1"][l]))
    scan_us = 1e3 * statistics.mean(scan_ms)
    attn_us = 1e3 * statistics.mean(attn_ms)
    topk_us = 1e3 * statistics.mean(topk_ms)
    n_cand = W_T - W_S - W_W
    scan_bytes = W_B * n_cand * SCAN_BYTES_PER_CAND
    attn_bytes = W_B * MAX_ROWS * W_HKV * ATTN_BYTES_PER_ROW_HEAD
    hbm_peak, peak_src = peaks()
    scan_gbs = scan_bytes / (scan_us * 1e-6) / 1e9
    attn_gbs = attn_bytes / (attn_us * 1e-6) / 1e9
    step_bytes = L * (scan_bytes + attn_bytes)
    step_gbs = step_bytes / (ms_per_step * 1e-3) / 1e9

    # ---- end to end through the API with host buffers -----------------------------------
    q_host = torch.empty(w.q.shape, dtype=w.q.dtype, pin_memory=True)
    k_host = torch.empty(w.newk.shape, dtype=w.newk.dtype, pin_memory=True)
    v_host = torch.empty(w.newv.shape, dtype=w.newv.dtype, pin_memory=True)
    o_host = torch.empty(w.out.shape, dtype=w.out.dtype, pin_memory=True)
    q_host.copy_(w.q)
    k_host.copy_(w.newk)
    v_host.copy_(w.newv)
    torch.cuda.synchronize()
    h2d = q_host.numel() * 2 + k_host.numel() * 2 + v_host.numel() * 2
    d2h = o_host.numel() * 4
    barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        with torch.cuda.stream(stream):
            w.q.copy_(q_host, non_blocking=True)
            w.newk.copy_(k_host, non_blocking=True)
            w.newv.copy_(v_host, non_blocking=True)
            graph.replay()
            o_host.copy_(w.out, non_blocking=True)
        stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / args.steps
    barrier()
    e2e_value = L * world / e2e_s

    if rank != 0:
        return
    gb = world * (L * (W_B * W_T * (2 * W_HKV * W_D + 4 * W_HKV + W_HKV * W_R // 2))) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int8/int4 storage, int32 scores, fp32 accumulate", "data": "synthetic",
        "config": config_dict(f"inputs larger than L2: {L} layers x {gb / world / L:.1f} GB resident, "
                              f"{step_bytes / 1e9:.2f} GB read per step", layers=L),
        "tokens_per_s": tokens_per_s, "hbm_gbs": step_gbs,
        "parallelism": "replicas only" if world > 1 else "single GPU",
        "kernel_us": {"score_select_int4": scan_us, "sparse_attend_int8": attn_us},
        "roofline": {"bound": "hbm", "achieved": scan_gbs, "peak": hbm_peak, "unit": "GB/s",
                     "frac": scan_gbs / hbm_peak, "traffic": measured_traffic("score_select"), "kernel": "score_select_kernel (scan + top-k)",
                     "peak_source": peak_src, "bytes_per_launch": scan_bytes,
                     "bytes_rule": f"{SCAN_BYTES_PER_CAND} B sketch row per candidate token x {W_B} x {n_cand}"},
        "roofline_attend": {"bound": "hbm", "achieved": attn_gbs, "peak": hbm_peak, "unit": "GB/s",
                            "frac": attn_gbs / hbm_peak, "traffic": measured_traffic("attend"), "bytes_per_launch": attn_bytes,
                            "bytes_rule": f"{ATTN_BYTES_PER_ROW_HEAD} B per row-head x {W_B} x {MAX_ROWS} x {W_HKV}"},
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * L * SketchWorkloadGPU.KERNELS_PER_LAYER,
        "clocks": clk.summary(), "device_status": status,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_block(args.cpu_budget)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--layers", type=int, default=W_L, help="distinct layers (16 for the workload; fewer only "
                    "for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

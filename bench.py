"""Batch-1 decode throughput of the 7B-shape bf16 stack on GB300.

One step = one token through all 32 layers (hidden 4096, 32 heads MHA, head
dim 128, FFN 11008) with the KV cache prefilled to 2047 positions, through the
library's C ABI (captured CUDA graph, fused plan of five kernels per layer).
Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline] [--layers L]
                  [--plan fused|four|three|persistent|unfused] [--eager]
                  [--no-pdl] [--no-l2-ahead] [--global-merge] [--lm-head VOCAB]
                  [--q4-publish]

--plan, --eager, --no-pdl, --no-l2-ahead and --global-merge select the
ablations of the default plan (five fused kernels a layer, CUDA graph,
programmatic dependent launch, L2 look-ahead, attention as one cluster per KV
head); --plan four folds the down GEMV into the gated-FFN kernel, --plan three
also attention and o-proj (each one launch of two phases).  --q4-publish (int4
workloads) has each GEMV input's producer publish its int8 codes once.

--impl reference times the fp64 CPU oracle on the host cores on the same
workload (the slow reference arm).  Under torchrun each rank decodes its own
replica (the path does not shard); rank 0 prints.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
# the kernel with the largest stream of the layer, per plan (index within the layer)
DOMINANT_KERNEL = {"three": 2, "four": 3, "fused": 3,  # gate/up (+ down when fused with it)
                   "headproj": 2, "headproj3": 2}
DOMINANT_NAME = {"three": "norm_gateup_swiglu_down_residual",
                 "four": "norm_gateup_swiglu_down_residual", "fused": "norm_gateup_swiglu",
                 "headproj": "norm_gateup_swiglu",
                 "headproj3": "norm_gateup_swiglu_down_residual"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="stack32_h4096_mha")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0,
                    help="override the layer count (small profiling cases only)")
    ap.add_argument("--plan", default="fused",
                    choices=["fused", "headproj", "headproj3", "four", "three", "persistent",
                             "unfused"],
                    help="fused five-kernel layer; attention + o-projection in one cluster "
                         "launch (headproj: four kernels, headproj3: with the two-phase FFN, "
                         "three); the four- or three-kernel layers with grid barriers; the "
                         "persistent per-token kernel; or the one-kernel-per-op ablation")
    ap.add_argument("--eager", action="store_true", help="launch eagerly instead of a CUDA graph")
    ap.add_argument("--no-pdl", action="store_true",
                    help="fused plan: no programmatic dependent launch between kernels")
    ap.add_argument("--no-l2-ahead", action="store_true",
                    help="fused plan: no L2 prefetch of the next kernel's bytes")
    ap.add_argument("--lm-head", type=int, default=0, metavar="VOCAB",
                    help="end every step with an LM head of this vocabulary and the greedy "
                         "token (not part of the headline workload, which has no LM head)")
    ap.add_argument("--global-merge", action="store_true",
                    help="fused plan: flat attention grid merged through global memory "
                         "instead of one cluster per KV head")
    ap.add_argument("--q4-publish", action="store_true",
                    help="int4 weights: the kernel that produces each GEMV input publishes its "
                         "int8 codes once, instead of every GEMV CTA quantizing the vector")
    return ap.parse_args()


def slowest_rank_ms(ms: float, world: int) -> float:
    """The step time of the whole job: the maximum over ranks (every rank calls this)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_tok_s(world: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput of `world` independent replicas, each decoding `steps` tokens."""
    return world * steps / (ms_max * 1e-3)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


# ---- accounting ---------------------------------------------------------------

def bytes_per_token(w, n_ctx_avg: float) -> dict:
    """Algorithmic bytes one token must move: all weights once, the KV read at the
    average context, the KV append."""
    weights = w.weight_bytes_per_layer() * w.n_layers
    kv_read = 2 * w.n_kv_heads * w.head_dim * 2 * n_ctx_avg * w.n_layers
    kv_append = 2 * w.n_kv_heads * w.head_dim * 2 * w.n_layers
    return {"weights": weights, "kv_read": kv_read, "kv_append": kv_append,
            "total": weights + kv_read + kv_append}


def kernel_bytes(w, kernel: int, n_ctx: int, plan: str = "fused") -> int:
    """Algorithmic bytes of one launch of a fused kernel (weights, norm vector,
    input and output vectors; for attention the K/V rows read and q, o).
    kernel: index within the layer of the five-kernel plan, or of the
    three-kernel plan (0 QKV, 1 attention + o-proj, 2 gate/up + down)."""
    H, F, hd, nq, nkv = w.hidden, w.ffn, w.head_dim, w.n_q_heads, w.n_kv_heads
    if plan in ("headproj", "headproj3") and kernel > 0:
        # 1: attention + o-projection; 2: gate/up (+ down); 3: down
        if kernel == 1:
            return kernel_bytes(w, 1, n_ctx) + kernel_bytes(w, 2, n_ctx)
        return kernel_bytes(w, kernel + 1, n_ctx, "four" if plan == "headproj3" else "fused")
    if plan == "four" and kernel == 3:
        return kernel_bytes(w, 3, n_ctx) + kernel_bytes(w, 4, n_ctx)
    if plan == "three" and kernel > 0:
        parts = (1, 2) if kernel == 1 else (3, 4)
        # the phases' shared vector (o, a) is written once and read once
        return sum(kernel_bytes(w, k, n_ctx) for k in parts)
    bpp = 2.0 if w.weight_fmt == "bf16" else 0.5 + 2.0 / 32  # bytes per weight
    if kernel == 0:
        return int(bpp * (nq + 2 * nkv) * hd * H) + 2 * H + 4 * H + 4 * nq * hd + 2 * 2 * nkv * hd
    if kernel == 1:
        return 2 * 2 * nkv * hd * n_ctx + 4 * nq * hd * 2
    if kernel == 2:
        return int(bpp * H * nq * hd) + 4 * nq * hd + 4 * H * 2
    if kernel == 3:
        return int(bpp * 2 * F * H) + 2 * H + 4 * H + 4 * F
    return int(bpp * H * F) + 4 * F + 4 * H * 2


def metric_name(w) -> str:
    if w.name == "stack32_h4096_mha":
        return "batch-1 decode tok/s (7B-shape bf16)"
    return f"batch-1 decode tok/s ({w.name}, {w.weight_fmt})"


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            for k in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
                if k in d:
                    return float(d[k]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _code_only(src: str) -> str:
    """C++ source without comments and blank lines (comment edits do not change a kernel)."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_sha() -> str:
    """Hash of the fused kernels' code (the sources the profiled traffic was taken on)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "transformer_layer_decode_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.startswith("kernels_fused") or f in ("common.cuh", "kernels.h", "phases.cuh"):
            h.update(_code_only(open(os.path.join(csrc, f)).read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", f"traffic_{kernel}_{workload}.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        if d.get("kernel_source_sha") == kernel_source_sha():
            return d.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


# ---- clocks -------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.windows = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        def reader():
            for line in self.proc.stdout:
                self.lines.append((time.time(), line.strip()))
        self.t = threading.Thread(target=reader, daemon=True)
        self.t.start()
        time.sleep(0.6)

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            inside = any(a - 0.05 <= ts <= b + 0.05 for a, b in self.windows)
            rows.append((inside, parts))
        use = [p for inside, p in rows if inside] or [p for _, p in rows]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in use if num(p[1]) is not None]
        mx = [num(p[2]) for p in use if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in use for n, v in zip(names, p[5:9]) if v == "Active"})
        pw = [num(p[3]) for p in use if num(p[3]) is not None]
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(use), "power_w_median": float(np.median(pw)) if pw else None}


# ---- the CPU oracle -------------------------------------------------------------

def oracle_for(w, host, max_ctx):
    from oracle import oracle as orc
    from transformer_layer_decode_gb300 import synth
    order = (synth.T_WQ, synth.T_WK, synth.T_WV, synth.T_WO, synth.T_WGATE, synth.T_WUP,
             synth.T_WDOWN)
    layers = []
    for lw in host["layers"]:
        if w.weight_fmt == "bf16":
            layers.append(dict(attn_norm=lw.attn_norm, ffn_norm=lw.ffn_norm,
                               w=[lw.mats[t] for t in order]))
        else:
            layers.append(dict(attn_norm=lw.attn_norm, ffn_norm=lw.ffn_norm,
                               q4=[lw.q4[t] for t in order]))
    st = orc.OracleStack(hidden=w.hidden, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads,
                         head_dim=w.head_dim, ffn=w.ffn, max_ctx=max_ctx, layers=layers,
                         rms_eps=w.rms_eps, rope_theta=w.rope_theta, q4=w.weight_fmt == "q4")
    for l, (k, v) in enumerate(host["kv"]):
        st.load_kv(l, k, v)
    return st


def oracle_cores() -> int:
    n = os.environ.get("OMP_NUM_THREADS")
    return int(n) if n and n.isdigit() else (os.cpu_count() or 1)


def time_oracle_tokens(w, host, budget_s: float, positions: int, max_tokens: int = 1 << 20):
    """Whole oracle tokens at the positions the timed region decodes (prefill
    to prefill + positions - 1, the cache rewound to the prefill at each wrap)
    until the time budget is spent, so the sample's size does not hang on the
    step count."""
    st = oracle_for(w, host, w.prefill + positions + 2)
    from transformer_layer_decode_gb300 import synth
    n, t_total = 0, 0.0
    while n < max_tokens and (n == 0 or t_total < budget_s):
        i = n % positions
        if i == 0:
            st.kv_len = w.prefill  # rewound: the rows past the prefill are written again
        x = synth.step_input(w, i)
        t0 = time.perf_counter()
        st.step(x, w.prefill + i)
        t_total += time.perf_counter() - t0
        n += 1
    return n, t_total


def host_workload(w):
    """Host copies of every layer's weights and KV prefill (seeded generator)."""
    from transformer_layer_decode_gb300 import synth
    host = {"layers": [], "kv": []}
    for l in range(w.n_layers):
        host["layers"].append(synth.layer_weights(w, l))
        host["kv"].append(synth.kv_bf16(w, l, w.prefill))
    return host


# ---- arms -----------------------------------------------------------------------

def run_reference(args, w, rank, world):
    if rank != 0:
        return None
    from oracle import oracle as orc
    orc.build()
    host = host_workload(w)
    # each step is one whole oracle token; if that would not fit in a few
    # minutes, a step is the first n layers of a token and the rate is scaled
    st = oracle_for(w, host, w.prefill + args.steps + args.warmup + 2)
    from transformer_layer_decode_gb300 import synth
    x0 = synth.step_input(w, 0)
    t0 = time.perf_counter()
    st.step(x0, w.prefill)
    t_tok = time.perf_counter() - t0
    budget = 150.0
    per_step = budget / max(1, args.steps + args.warmup)
    n_layers = w.n_layers if t_tok <= per_step else max(1, int(w.n_layers * per_step / t_tok))
    st = oracle_for(w, host, w.prefill + 2)
    import ctypes
    cur = np.ascontiguousarray(x0, dtype=np.float64)
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        x = cur
        for l in range(n_layers):
            x = st.layer_step(l, x, w.prefill)  # each layer feeds the next, as in a token
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
    t_step = float(np.sum(times)) / args.steps
    sec_per_token = t_step * w.n_layers / n_layers
    value = 1.0 / sec_per_token
    sample = (f"{n_layers} of {w.n_layers} layers per step at pos {w.prefill}, "
              f"scaled to whole tokens" if n_layers < w.n_layers else
              f"whole tokens at pos {w.prefill}")
    return {
        "impl": "reference", "metric": metric_name(w),
        "value": value, "unit": "tok/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "layers": w.n_layers, "hidden": w.hidden,
                   "heads": f"{w.n_q_heads}/{w.n_kv_heads}", "head_dim": w.head_dim,
                   "ffn": w.ffn, "prefill": w.prefill, "batch": 1,
                   "parallelism": "single-gpu", "plan": "fp64 CPU oracle (unfused chain)"},
        "cpu_baseline": {"value": value, "unit": "tok/s", "cores": oracle_cores(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_ours(args, w, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    from transformer_layer_decode_gb300 import build as tld_build
    from transformer_layer_decode_gb300 import dec, synth, workload
    if world > 1:  # one rank compiles (if anything is stale); the others wait for it
        if rank == 0:
            tld_build.build()
        dist.barrier()
    tld_build.build()
    dev = torch.device("cuda", local_rank)
    K, W = args.steps, args.warmup
    max_ctx = w.prefill + max(K, W) + 2
    want_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    unfused = args.plan == "unfused"
    persistent = args.plan == "persistent"
    d, host = workload.make_decoder(w, max_ctx=max_ctx, keep_host=want_cpu, unfused=unfused,
                                    persistent=persistent, graph=not args.eager,
                                    pdl=not args.no_pdl, l2_ahead=not args.no_l2_ahead,
                                    cluster_attn=not args.global_merge, three=args.plan == "three",
                                    four=args.plan in ("four", "headproj3"),
                                    attn_oproj=args.plan in ("headproj", "headproj3"),
                                    q4_publish=args.q4_publish)
    if args.lm_head:
        nw, Wlm = synth.lm_head(w, args.lm_head)
        d.load_lm_head(nw, Wlm)
        tok_out = torch.empty(1, dtype=torch.int32, device=dev)
        d.set_token_out(tok_out)
    info = d.info()
    H = w.hidden
    xs = torch.from_numpy(workload.step_inputs(w, max(K, W))).to(dev)
    out = torch.empty(H, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    # warm-up, then rewind the cache to the prefill
    for s in range(W):
        d.step(xs[s], w.prefill + s, out)
    d.sync_status()
    d.truncate_kv(w.prefill)

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid).replace("GPU-", "")
    except Exception:
        uuid = str(local_rank)
    clocks = ClockSampler(uuid)
    clocks.start()

    # ---- timed region: K steps, inputs resident in HBM -------------------------
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    tw0 = time.time()
    ev0.record(stream)
    for s in range(K):
        d.step(xs[s], w.prefill + s, out)
    ev1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    barrier()
    clocks.mark(tw0, tw1)
    d.sync_status()
    ms = slowest_rank_ms(ev0.elapsed_time(ev1), world)

    # ---- end to end: host input -> device, step, device -> host each step ------
    d.truncate_kv(w.prefill)
    host_in = torch.from_numpy(workload.step_inputs(w, K)).pin_memory()
    host_out = torch.empty(K, H, dtype=torch.float32).pin_memory()
    emb = torch.empty(H, dtype=torch.float32, device=dev)
    barrier()
    torch.cuda.synchronize()
    tw0 = time.time()
    ev0.record(stream)
    for s in range(K):
        emb.copy_(host_in[s], non_blocking=True)
        d.step(emb, w.prefill + s, out)
        host_out[s].copy_(out, non_blocking=True)
    ev1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    barrier()
    clocks.mark(tw0, tw1)
    ms_e2e = slowest_rank_ms(ev0.elapsed_time(ev1), world)
    assert np.all(np.isfinite(host_out.numpy())), "non-finite decode output"

    # ---- dominant kernel alone: back to back over all layers' weights ----------
    n_ctx = w.prefill + K  # KV length after the timed steps
    dom = DOMINANT_KERNEL.get(args.plan, 3)
    kb = kernel_bytes(w, dom, n_ctx, args.plan)
    peak, peak_kind = measured_peaks()
    if persistent:
        # one kernel per step: its launches are exactly the timed region's steps
        kb = bytes_per_token(w, w.prefill + (K + 1) / 2.0)["total"]
        k_ms = ms / K
        achieved = kb / (k_ms * 1e-3) / 1e9
    elif not unfused:
        d.launch_kernel(dom, 0, w.n_layers)  # warm
        reps = 3
        torch.cuda.synchronize()
        tw0 = time.time()
        ev0.record(stream)
        for _ in range(reps):
            d.launch_kernel(dom, 0, w.n_layers)
        ev1.record(stream)
        torch.cuda.synchronize()
        tw1 = time.time()
        d.sync_status()
        clocks.mark(tw0, tw1)
        k_ms = ev0.elapsed_time(ev1) / (reps * w.n_layers)
        achieved = kb / (k_ms * 1e-3) / 1e9
    else:
        k_ms, achieved = None, None
    clocks.stop()
    kname = ("token_persistent" if persistent else DOMINANT_NAME.get(args.plan, "none"))
    traffic = profiled_traffic(w.name, kname) if args.plan in DOMINANT_NAME else None

    tok_s = replica_tok_s(world, K, ms)
    tok_s_e2e = replica_tok_s(world, K, ms_e2e)
    bpt = bytes_per_token(w, w.prefill + (K + 1) / 2.0)
    if args.lm_head:
        lm_bytes = 2 * args.lm_head * (w.hidden + 1)
        bpt = {**bpt, "lm_head": lm_bytes, "total": bpt["total"] + lm_bytes}

    result = {
        "metric": metric_name(w),
        "value": tok_s, "unit": "tok/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.weight_fmt == "bf16" else "int4/int8",
        "data": "synthetic",
        "config": {"workload": w.name, "layers": w.n_layers, "hidden": w.hidden,
                   "heads": f"{w.n_q_heads}/{w.n_kv_heads}", "head_dim": w.head_dim,
                   "ffn": w.ffn, "prefill": w.prefill, "batch": 1,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "plan": ", ".join([args.plan, "eager" if args.eager else "CUDA graph"]
                                     + (["no PDL"] if args.no_pdl else [])
                                     + (["no L2 look-ahead"] if args.no_l2_ahead else [])
                                     + (["global-merge attention"] if args.global_merge else [])
                                     + (["int8 inputs published by their producers"]
                                        if args.q4_publish else [])),
                   "kernels_per_layer": info.kernels_per_layer,
                   "kernels_per_token": info.kernels_per_token + (1 if args.lm_head else 0),
                   "lm_head_vocab": args.lm_head or None,
                   "attn_ctas": info.attn_grid, "attn_cluster": info.attn_cluster,
                   "l2": "no flush: each step streams %.1f GB of weights + KV (> 129 MB L2)"
                         % (bpt["total"] / 1e9)},
        "hbm": {"bytes_per_token": bpt["total"], "achieved_gbs": bpt["total"] * tok_s / world / 1e9,
                "peak_gbs": peak, "peak_kind": peak_kind,
                "frac": bpt["total"] * tok_s / world / 1e9 / peak},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak if achieved else None, "traffic": traffic,
                     "kernel": kname,
                     "bytes_per_launch": kb,
                     "avg_launch_ms": k_ms, "peak_kind": peak_kind},
        "e2e": {"value": tok_s_e2e, "unit": "tok/s", "h2d_bytes_per_step": 4 * H,
                "d2h_bytes_per_step": 4 * H},
        "gpu_launches": (info.kernels_per_token + (1 if args.lm_head else 0)) * K,
        "clocks": clocks.summary(),
    }
    d.close()
    if want_cpu:
        from oracle import oracle as orc
        orc.build()
        n, t = time_oracle_tokens(w, host, budget_s=15.0, positions=K)
        result["cpu_baseline"] = {"value": n / t, "unit": "tok/s", "cores": oracle_cores(),
                                  "kind": "oracle",
                                  "sample": f"{n} whole tokens at the timed positions "
                                            f"{w.prefill}..{w.prefill + K - 1} (the cache rewound "
                                            f"at each wrap; {t:.1f} s of CPU work)"}
    return result if rank == 0 else None


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    from transformer_layer_decode_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = w.small(n_layers=args.layers, name=f"{w.name}_{args.layers}layers")
    if args.impl == "reference":
        res = run_reference(args, w, rank, world)
    else:
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl")
        res = run_ours(args, w, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the G-LRD decode-attention hot path on one node.

One step = one decode step of one attention layer over a latent KV cache already
resident in HBM: append the new token's K/V latents (quantising them for int4
caches), prepare the query, run the decode-attention kernel over all cached
tokens, and merge the split-T partials. The default workload is the Llama-2-7B
RoPE layer with fp16 latents at batch 1 and T = 4096 tokens.

Prints ONE JSON line (rank 0). ``--impl reference`` times the float64 CPU oracle
instead, on a bounded sample of the same workload.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn latency µs & effective KV GB/s at T=4K–64K; % of roofline"

# name -> (workload in synthetic.gen, T override)
WORKLOADS = {
    "tiny-fp32-b1-t512": ("TINY_FP32", None),
    "llama2-7b-rope-fp16-b1-t4k": ("ROPE_FP16", None),
    "llama2-7b-rope-bf16-b8-t16k": ("ROPE_BF16", 16384),
    "llama2-7b-rope-bf16-b8-t32k": ("ROPE_BF16", None),
    "llama2-7b-absorbed-fp16-b4-t64k": ("ABSORBED_FP16", None),
    "llama2-7b-rope-int4-hadamard-b4-t64k": ("ROPE_INT4", None),
}
DEFAULT_WORKLOAD = "llama2-7b-rope-fp16-b1-t4k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------
# Algorithmic work of one step (bytes the path must move, flops it must do)
# ---------------------------------------------------------------------------

def kv_bytes_dense(layers, kv_heads, head_dim, tokens, bytes_per_elem):
    """Uncompressed KV size 2 * L * H_kv * d * T * bytes (the formula of the Shard write-up, section 1)."""
    return 2 * layers * kv_heads * head_dim * tokens * bytes_per_elem


def latent_bytes_per_token(cfg):
    """K + V latent bytes one token occupies across all groups of one layer."""
    if cfg.latent_dtype == "int4":
        return cfg.n_groups * ((cfg.rank // 2) * 2 + 2 * 2)  # codes + one fp16 scale each for K and V
    elt = 4 if cfg.latent_dtype == "f32" else 2
    return cfg.n_groups * 2 * cfg.rank * elt


def step_work(cfg):
    """Algorithmic bytes and flops of one decode step of the workload."""
    B, T = cfg.batch, cfg.T
    bk_elt = 4 if cfg.bk_dtype == "f32" else 2
    bk_bytes = cfg.n_groups * cfg.rank * cfg.group_size * cfg.head_dim * bk_elt
    latent = B * T * latent_bytes_per_token(cfg)
    decode_bytes = latent + bk_bytes
    if cfg.mode == "rope":
        flops = 2 * B * T * cfg.n_groups * cfg.rank * cfg.group_size * cfg.head_dim
    else:
        flops = 2 * B * T * cfg.n_heads * cfg.rank  # q' . h_k per head and token
    flops += 2 * B * T * cfg.n_heads * cfg.rank     # p . H_v
    append_bytes = B * latent_bytes_per_token(cfg)
    dense_equiv = B * kv_bytes_dense(1, cfg.n_heads, cfg.head_dim, T, 2)
    return {"decode_bytes": decode_bytes, "latent_bytes": latent, "bk_bytes": bk_bytes, "flops": flops,
            "append_bytes": append_bytes, "dense_fp16_kv_bytes": dense_equiv}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def roofline_for(cfg, work, kernel_ms, peaks, peaks_src, long_step):
    hbm = float(peaks["hbm_gbs"])
    tc = float(peaks["bf16_tflops_sustained" if long_step else "bf16_tflops"])  # fp16 = bf16 nominal rate
    t_hbm = work["decode_bytes"] / (hbm * 1e9)
    t_tc = work["flops"] / (tc * 1e12) if cfg.mode == "rope" else 0.0
    sec = kernel_ms / 1e3
    if t_tc > t_hbm:
        ach = work["flops"] / sec / 1e12
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": tc, "unit": "TFLOP/s",
                "frac": round(ach / tc, 4), "traffic": None,
                "peak_source": f"{'bf16_tflops_sustained' if long_step else 'bf16_tflops'} of {peaks_src}"}
    ach = work["decode_bytes"] / sec / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
            "traffic": None, "peak_source": f"hbm_gbs of {peaks_src}"}


# ---------------------------------------------------------------------------
# DRAM traffic of the decode kernel, from a recorded ncu capture
# ---------------------------------------------------------------------------

CSRC = os.path.join(ROOT, "rank_kv_cache_gb300", "csrc")
KERNEL_SOURCES = {
    "decode_tc_kernel": ("decode_tc.cu", "tc_ptx.cuh"),
    "decode_abs_kernel": ("decode_abs.cu", "tc_ptx.cuh"),
    "decode_simt_kernel": ("decode_simt.cu",),
}
COMMON_SOURCES = ("split_merge.cuh", "internal.h", "common.cuh")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def _code_only(text):
    """Source text without comments and blank-space differences (what the compiler sees)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel):
    """Hash of the code (comments and layout ignored) of the files a decode kernel is compiled
    from, first 16 hex digits."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel] + COMMON_SOURCES:
        with open(os.path.join(CSRC, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload, kernel, cfg):
    """dram__bytes_read.sum + dram__bytes_write.sum per launch of `kernel` on this workload,
    from the recorded capture of the same kernel source; scaled by tokens processed when the
    capture ran a smaller batch or T. None when no capture matches the current source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        entries = json.load(f).get("entries", [])
    src = kernel_source_hash(kernel)
    for e in entries:
        if e.get("workload") == workload and e.get("kernel") == kernel and e.get("source_sha256") == src:
            scale = (cfg.batch * cfg.T) / (e["batch"] * e["tokens"])
            return int(round(e["dram_bytes"] * scale))
    return None


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, dist=None, device="cpu"):
    """The largest value of x across the ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(world, bytes_per_rank_step, ms_per_step):
    """Whole-job GB/s of independent replicas: every rank moves bytes_per_rank_step per step and the
    step takes as long as the slowest rank (weak scaling)."""
    return world * bytes_per_rank_step / 1e9 / (ms_per_step / 1e3)


class GpuWorkload:
    """Device-resident workload: cache filled through the append kernel, per-step inputs."""

    def __init__(self, cfg, device):
        import torch
        from rank_kv_cache_gb300 import palu as P
        from synthetic import gen
        self.cfg, self.dev = cfg, device
        inp = gen.make_inputs(cfg)
        B, T = cfg.batch, cfg.T
        lat = cfg.latent_dtype
        self.attn = P.PaluAttention(gen.storage_round(inp["bk"], cfg.bk_dtype).to(device), n_heads=cfg.n_heads,
                                    head_dim=cfg.head_dim, group_size=cfg.group_size, rank_k=cfg.rank,
                                    rank_v=cfg.rank, latent_dtype=lat, q_dtype=cfg.q_dtype, mode=cfg.mode,
                                    rope_theta=cfg.theta, max_batch=B, max_tokens=T)
        self.cache = P.LatentCache(B, T, cfg.n_groups, cfg.rank, cfg.rank, lat, device=device)
        src_dt = "f32" if lat == "int4" else lat
        hk = gen.storage_round(inp["hk"], src_dt).to(device)
        hv = gen.storage_round(inp["hv"], src_dt).to(device)
        zero = torch.zeros(B, dtype=torch.int32, device=device)
        self.attn.append(self.cache, hk, hv, zero)            # prefill the cache (not timed)
        self.hk_new = hk[:, T - 1:T].contiguous()             # the step's new token (rewritten at slot T-1)
        self.hv_new = hv[:, T - 1:T].contiguous()
        del hk, hv
        self.slot = torch.full((B,), T - 1, dtype=torch.int32, device=device)
        self.seq = torch.full((B,), T, dtype=torch.int32, device=device)
        self.q = gen.storage_round(inp["q"], cfg.q_dtype).to(device)
        self.out = torch.empty((B, cfg.n_heads, cfg.rank), dtype=torch.float32, device=device)
        self.lse = torch.empty((B, cfg.n_heads), dtype=torch.float32, device=device)
        torch.cuda.synchronize()

    def step(self):
        self.attn.append(self.cache, self.hk_new, self.hv_new, self.slot)
        self.attn.decode(self.q, self.cache, self.seq, max_seq_len=self.cfg.T, out=self.out, lse=self.lse)

    @property
    def launches_per_step(self):
        # one append launch (K and V together) + the decode call's own launches: the split
        # merge runs inside the decode kernel; the absorbed and CUDA-core kernels add a
        # query-preparation launch
        kernel, _, launches = self.attn.plan(self.cfg.T, self.cfg.batch, self.cfg.T)
        return 1 + launches

    @property
    def kernel_name(self):
        from rank_kv_cache_gb300 import palu as P
        kernel = self.attn.plan(self.cfg.T, self.cfg.batch, self.cfg.T)[0]
        return {P.PALU_KERNEL_TC_ROPE: "decode_tc_kernel", P.PALU_KERNEL_TMA_ABSORBED: "decode_abs_kernel",
                P.PALU_KERNEL_SIMT: "decode_simt_kernel"}[kernel]


def run_gpu(args, cfg, name):
    import torch
    from rank_kv_cache_gb300 import palu as P
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    wl = GpuWorkload(cfg, dev)
    work = step_work(cfg)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # > 2x the 129 MB L2
    W, K = args.warmup, args.steps

    for _ in range(W):
        flush.zero_()
        wl.step()
    torch.cuda.synchronize()
    wl.attn.check_device()

    # device-timed steps (inputs resident in HBM), L2 flushed before every step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    P.check(P.palu_attn_trace_enable(wl.attn.handle, 1))
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t0 = time.perf_counter()
        for i in range(K):
            flush.zero_()
            ev[i][0].record()
            wl.step()
            ev[i][1].record()
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
    if dist:
        dist.barrier()
    st, n_tr, tr_ms = P.palu_attn_trace_read(wl.attn.handle)
    P.check(st)
    P.palu_attn_trace_enable(wl.attn.handle, 0)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    tot_ms = max_over_ranks(sum(step_ms), dist, dev)
    ms_per_step = tot_ms / K
    kernel_ms = tr_ms / max(n_tr, 1)
    wl.attn.check_device()

    # end-to-end through the public API: pinned host inputs in, result back to host, every step
    q_h = wl.q.cpu().pin_memory()
    hk_h, hv_h = wl.hk_new.cpu().pin_memory(), wl.hv_new.cpu().pin_memory()
    out_h = torch.empty(wl.out.shape, dtype=torch.float32).pin_memory()
    lse_h = torch.empty(wl.lse.shape, dtype=torch.float32).pin_memory()
    h2d = q_h.numel() * q_h.element_size() + hk_h.numel() * hk_h.element_size() + hv_h.numel() * hv_h.element_size()
    d2h = out_h.numel() * 4 + lse_h.numel() * 4
    Ke = min(K, 200)
    e2e_ms = []
    for i in range(Ke):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        wl.q.copy_(q_h, non_blocking=True)
        wl.hk_new.copy_(hk_h, non_blocking=True)
        wl.hv_new.copy_(hv_h, non_blocking=True)
        wl.step()
        out_h.copy_(wl.out, non_blocking=True)
        lse_h.copy_(wl.lse, non_blocking=True)
        b.record()
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e_step = max_over_ranks(statistics.mean(e2e_ms), dist, dev)

    peaks, peaks_src = load_peaks()
    roof = roofline_for(cfg, work, kernel_ms, peaks, peaks_src, long_step=ms_per_step > 10.0)
    roof["kernel"] = wl.kernel_name
    roof["traffic"] = recorded_traffic(name, wl.kernel_name, cfg)
    result = {
        "metric": METRIC,
        "value": round(job_throughput_gbs(world, work["decode_bytes"], ms_per_step), 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_per_step, 6),
        "latency_us": round(ms_per_step * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.latent_dtype,
        "data": "synthetic (seeded spectrum-decay weights, Gaussian activations and queries)",
        "config": {"workload": name, "batch": cfg.batch, "tokens": cfg.T, "heads": cfg.n_heads,
                   "head_dim": cfg.head_dim, "group_size": cfg.group_size, "rank": cfg.rank,
                   "latent_dtype": cfg.latent_dtype, "mode": cfg.mode, "hadamard": cfg.hadamard,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed (512 MB write) before every timed step",
                   "bytes_per_step": work["decode_bytes"], "flops_per_step": work["flops"],
                   "dense_fp16_kv_bytes_per_step": work["dense_fp16_kv_bytes"]},
        "dense_equiv_gbs": round(job_throughput_gbs(world, work["dense_fp16_kv_bytes"], ms_per_step), 1),
        "roofline": roof,
        "kernel_us": round(kernel_ms * 1e3, 2),
        "kernel_launches_traced": n_tr,
        "e2e": {"value": round(job_throughput_gbs(world, work["decode_bytes"], e2e_step), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_step, 6),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke},
        "gpu_launches": wl.launches_per_step * K,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 4),
    }
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(cfg, work, budget_s=args.cpu_seconds)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return result if rank == 0 else None


# ---------------------------------------------------------------------------
# CPU oracle: baseline leg and reference arm
# ---------------------------------------------------------------------------

def _blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


class OracleSample:
    """The oracle on storage-rounded inputs of the workload, one (batch, head) at a time."""

    def __init__(self, cfg):
        import numpy as np
        from oracle import palu_oracle as O
        from synthetic import gen
        self.O, self.np, self.cfg = O, np, cfg
        inp = gen.make_inputs(cfg)
        if cfg.latent_dtype == "int4":
            ck, sk = O.quantize_int4(inp["hk"])
            cv, sv = O.quantize_int4(inp["hv"])
            self.hk = O.dequant_int4(O.pack_int4(ck), sk).astype(np.float32)
            self.hv = O.dequant_int4(O.pack_int4(cv), sv).astype(np.float32)
        else:
            self.hk = gen.storage_round(inp["hk"], cfg.latent_dtype).float().numpy()
            self.hv = gen.storage_round(inp["hv"], cfg.latent_dtype).float().numpy()
        self.q = gen.storage_round(inp["q"], cfg.q_dtype).double().numpy()
        self.bk = gen.storage_round(inp["bk"], cfg.bk_dtype).double().numpy()
        self.seq = np.full(cfg.batch, cfg.T)
        self.heads = [(b, i) for b in range(cfg.batch) for i in range(cfg.n_heads)]

    def run(self, heads):
        c = self.cfg
        return self.O.decode(self.q, self.hk, self.hv, self.bk, self.seq, c.group_size, mode=c.mode, theta=c.theta,
                             heads=heads)


def cpu_baseline(cfg, work, budget_s=12.0):
    """Time the oracle as it stands on this host's cores over a bounded sample of the workload."""
    sample = OracleSample(cfg)
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s:
        h = sample.heads[done % len(sample.heads)]
        sample.run([h])
        done += 1
    el = time.perf_counter() - t0
    frac = done / len(sample.heads)
    return {"value": round(work["decode_bytes"] * frac / el / 1e9, 4), "unit": "GB/s", "cores": _blas_threads(),
            "kind": "oracle", "seconds": round(el, 2),
            "sample": f"{done} single-head decodes cycling over the workload's {len(sample.heads)} (batch, head) "
                      f"pairs, all {cfg.T} tokens each, float64 NumPy"}


def run_reference(args, cfg, name):
    world, rank, _ = _dist()
    if rank != 0:
        return None
    work = step_work(cfg)
    sample = OracleSample(cfg)
    per_step = sample.heads[:cfg.group_size]  # one G-LRD group of one batch row, all T tokens
    frac = len(per_step) / len(sample.heads)
    for _ in range(args.warmup):
        sample.run(per_step)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        sample.run(per_step)
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    val = round(work["decode_bytes"] * frac / (ms / 1e3) / 1e9, 4)
    desc = f"{len(per_step)} heads (one group, batch row 0) of the workload per step, float64 NumPy"
    return {"metric": METRIC, "value": val, "unit": "GB/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "batch": cfg.batch, "tokens": cfg.T, "sample": desc},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": _blas_threads(), "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (profiling runs)")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's T (profiling runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    from synthetic import gen
    base, T = WORKLOADS[args.workload]
    cfg = getattr(gen, base) if T is None else getattr(gen, base).with_(T=T)
    if args.batch is not None:
        cfg = cfg.with_(batch=args.batch)
    if args.tokens is not None:
        cfg = cfg.with_(T=args.tokens)
    res = run_reference(args, cfg, args.workload) if args.impl == "reference" else run_gpu(args, cfg, args.workload)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the G-LRD decode-attention hot path on one node.

One step = one decode step of one attention layer over a latent KV cache already
resident in HBM: append the new token's K/V latents (quantising them for int4
caches), prepare the query, run the decode-attention kernel over all cached
tokens, and merge the split-T partials. The headline workload is the Llama-2-7B
RoPE layer with int4 latents (Hadamard-folded factors) at batch 4 and T = 65536;
``per_config`` in the same line times every other workload of the benchmark
(T = 512 to 64K) the same way, each with its own roofline fraction and oracle
baseline.

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
import tempfile
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
DEFAULT_WORKLOAD = "llama2-7b-rope-int4-hadamard-b4-t64k"
PER_CONFIG_ORDER = ("tiny-fp32-b1-t512", "llama2-7b-rope-fp16-b1-t4k", "llama2-7b-rope-bf16-b8-t16k",
                    "llama2-7b-rope-bf16-b8-t32k", "llama2-7b-absorbed-fp16-b4-t64k",
                    "llama2-7b-rope-int4-hadamard-b4-t64k")
SINGLE_CORE_ORACLE = ("tiny-fp32-b1-t512", "llama2-7b-rope-fp16-b1-t4k")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def config_of(name, batch=None, tokens=None):
    from synthetic import gen
    base, T = WORKLOADS[name]
    cfg = getattr(gen, base) if T is None else getattr(gen, base).with_(T=T)
    if batch is not None:
        cfg = cfg.with_(batch=batch)
    if tokens is not None:
        cfg = cfg.with_(T=tokens)
    return cfg


# ---------------------------------------------------------------------------
# Algorithmic work of one step (bytes the path must move, flops it must do)
# ---------------------------------------------------------------------------

def kv_bytes_dense(layers, kv_heads, head_dim, tokens, bytes_per_elem):
    """Uncompressed KV size 2 * L * H_kv * d * T * bytes (the formula of the Shard write-up, section 1)."""
    return 2 * layers * kv_heads * head_dim * tokens * bytes_per_elem


def latent_bytes_per_token(cfg):
    """K + V latent bytes one token occupies across all groups of one layer."""
    def side(dtype):
        if dtype == "int4":
            return cfg.rank // 2 + 2                         # codes + one fp16 scale
        return cfg.rank * (4 if dtype == "f32" else 2)
    return cfg.n_groups * (side(cfg.latent_dtype) + side(cfg.value_dtype))


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


GB300_SMS = 152
FP32_LANES_PER_SM = 128


def alu_peak_tflops(peaks):
    """fp32 FMA peak of the CUDA cores: 152 SMs x 128 lanes x 2 flops x the maximum SM clock."""
    return GB300_SMS * FP32_LANES_PER_SM * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12


def roofline_for(cfg, work, kernel_ms, peaks, peaks_src, long_step):
    """The slowest of latent bytes over HBM, (RoPE) rebuild flops over the tensor peak and
    (absorbed) score and p.H_v flops over the CUDA cores' fp32 peak bounds the decode kernel;
    achieved = that resource's algorithmic work / the kernel's duration."""
    hbm = float(peaks["hbm_gbs"])
    tc_key = "bf16_tflops_sustained" if long_step else "bf16_tflops"
    tc = float(peaks[tc_key])  # fp16 = bf16 nominal rate
    t_hbm = work["decode_bytes"] / (hbm * 1e9)
    t_tc = work["flops"] / (tc * 1e12) if cfg.mode == "rope" else 0.0
    sec = kernel_ms / 1e3
    alu = alu_peak_tflops(peaks)
    t_alu = work["flops"] / (alu * 1e12) if cfg.mode != "rope" else 0.0
    if t_alu > t_hbm:
        ach = work["flops"] / sec / 1e12
        return {"bound": "alu", "achieved": round(ach, 2), "peak": round(alu, 1), "unit": "TFLOP/s",
                "frac": round(ach / alu, 4), "traffic": None, "roofline_us": round(t_alu * 1e6, 2),
                "peak_source": f"152 SMs x 128 fp32 lanes x 2 x sm_max_mhz of {peaks_src}"}
    if t_tc > t_hbm:
        ach = work["flops"] / sec / 1e12
        return {"bound": "tensor", "achieved": round(ach, 2), "peak": tc, "unit": "TFLOP/s",
                "frac": round(ach / tc, 4), "traffic": None, "roofline_us": round(t_tc * 1e6, 2),
                "peak_source": f"{tc_key} of {peaks_src}"}
    ach = work["decode_bytes"] / sec / 1e9
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
            "traffic": None, "roofline_us": round(t_hbm * 1e6, 2), "peak_source": f"hbm_gbs of {peaks_src}"}


def pct(xs, q):
    """q-th percentile (0..100) of a non-empty list, linear interpolation."""
    s = sorted(xs)
    if len(s) == 1:
        return s[0]
    k = (len(s) - 1) * q / 100.0
    lo, hi = int(math.floor(k)), int(math.ceil(k))
    return s[lo] + (s[hi] - s[lo]) * (k - lo)


def stats_us(ms_list):
    us = [m * 1e3 for m in ms_list]
    return {"median": round(pct(us, 50), 2), "p10": round(pct(us, 10), 2), "p90": round(pct(us, 90), 2),
            "mean": round(statistics.mean(us), 2), "n": len(us)}


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
    """Device-resident workload: the latent cache drawn on the device and filled through the
    append kernel one batch row at a time, plus the per-step inputs."""

    def __init__(self, cfg, device, max_position=0, flags=0):
        import torch
        from rank_kv_cache_gb300 import palu as P
        from synthetic import gen
        self.cfg, self.dev, self.P = cfg, device, P
        B, T, n_g, r = cfg.batch, cfg.T, cfg.n_groups, cfg.rank
        lat = cfg.latent_dtype
        fac, _ = gen.factors(cfg)
        self.bk_host = gen.storage_round(fac["k"][1], cfg.bk_dtype)
        self.attn = P.PaluAttention(self.bk_host.to(device), n_heads=cfg.n_heads, head_dim=cfg.head_dim,
                                    group_size=cfg.group_size, rank_k=r, rank_v=r, latent_dtype=lat,
                                    q_dtype=cfg.q_dtype, mode=cfg.mode, rope_theta=cfg.theta, max_batch=B,
                                    max_tokens=T, max_position=max_position, v_dtype=cfg.value_dtype, flags=flags)
        self.cache = P.LatentCache(B, T, n_g, r, r, lat, device=device, v_dtype=cfg.value_dtype)
        src_dt = "f32" if lat in ("int4", "f32") else lat
        tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[src_dt]
        zero = torch.zeros(1, dtype=torch.int32, device=device)
        new_k, new_v = [], []
        self.sample_hk = self.sample_hv = None
        row_bytes_k = self.cache.hk[0].numel() * self.cache.hk.element_size()
        row_bytes_v = self.cache.hv[0].numel() * self.cache.hv.element_size()
        for b, (zk, zv) in enumerate(zip(gen.latent_rows_torch(cfg, device, "k"),
                                         gen.latent_rows_torch(cfg, device, "v"))):
            if b == 0:   # the oracle's sample: group 0 of batch row 0, unrounded float32
                self.sample_hk = zk[:, 0, :].cpu().numpy()
                self.sample_hv = zv[:, 0, :].cpu().numpy()
            hk, hv = zk.to(tdt)[None], zv.to(tdt)[None]
            new_k.append(hk[:, T - 1:T].clone())
            new_v.append(hv[:, T - 1:T].clone())
            c = self.cache.c_struct()
            c.hk += b * row_bytes_k
            c.hv += b * row_bytes_v
            if lat == "int4":
                c.k_scale += b * T * n_g * 2
            if cfg.value_dtype == "int4":
                c.v_scale += b * T * n_g * 2
            P.check(P.palu_append_latents(self.attn.handle, c, hk.data_ptr(), hv.data_ptr(), P.DTYPES[src_dt],
                                          zero.data_ptr(), 1, T, int(torch.cuda.current_stream().cuda_stream)),
                    "prefill append")
            del zk, zv, hk, hv
        torch.cuda.synchronize()
        self.hk_new = torch.cat(new_k).contiguous()       # the step's new token (rewritten at slot T-1)
        self.hv_new = torch.cat(new_v).contiguous()
        self.slot = torch.full((B,), T - 1, dtype=torch.int32, device=device)
        self.seq = torch.full((B,), T, dtype=torch.int32, device=device)
        self.q_host = gen.draw_query(cfg)
        self.q = gen.storage_round(self.q_host, cfg.q_dtype).to(device)
        self.out = torch.empty((B, cfg.n_heads, r), dtype=torch.float32, device=device)
        self.lse = torch.empty((B, cfg.n_heads), dtype=torch.float32, device=device)
        torch.cuda.synchronize()

    def step(self):
        self.attn.append(self.cache, self.hk_new, self.hv_new, self.slot)
        self.attn.decode(self.q, self.cache, self.seq, max_seq_len=self.cfg.T, out=self.out, lse=self.lse)

    def plan(self):
        return self.attn.plan(self.cfg.T, self.cfg.batch, self.cfg.T)

    @property
    def launches_per_step(self):
        # one append launch (K and V together) + the decode call's own launches: the split
        # merge runs inside the decode kernel; the absorbed and CUDA-core kernels add a
        # query-preparation launch
        return 1 + self.plan()[2]

    @property
    def kernel_name(self):
        P = self.P
        return {P.PALU_KERNEL_TC_ROPE: "decode_tc_kernel", P.PALU_KERNEL_TMA_ABSORBED: "decode_abs_kernel",
                P.PALU_KERNEL_SIMT: "decode_simt_kernel"}[self.plan()[0]]

    def oracle_sample(self):
        return OracleSample(self.cfg, self.sample_hk, self.sample_hv, self.q_host, self.bk_host)

    def close(self):
        self.attn.close()


def timed_steps(wl, n, flush, clock_gpu=None):
    """n device-timed steps, L2 flushed before each: (step ms list, decode-kernel ms list, clocks)."""
    import torch
    P = wl.P
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    P.check(P.palu_attn_trace_enable(wl.attn.handle, 1))
    torch.cuda.synchronize()
    with ClockSampler(clock_gpu if clock_gpu is not None else 0) as clk:
        for i in range(n):
            flush.zero_()
            ev[i][0].record()
            wl.step()
            ev[i][1].record()
        torch.cuda.synchronize()
    st, kms = P.palu_attn_trace_times(wl.attn.handle)
    P.check(st, "palu_attn_trace_times")
    P.check(P.palu_attn_trace_enable(wl.attn.handle, 0))
    wl.attn.check_device()
    return [a.elapsed_time(b) for a, b in ev], kms, clk.summary()


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
    st, kernel_ms_list = P.palu_attn_trace_times(wl.attn.handle)
    P.check(st)
    P.palu_attn_trace_enable(wl.attn.handle, 0)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    tot_ms = max_over_ranks(sum(step_ms), dist, dev)
    ms_per_step = tot_ms / K
    kernel_ms = statistics.mean(kernel_ms_list) if kernel_ms_list else float("nan")
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
    roof["duration"] = "mean decode-kernel launch over the timed steps (CUDA events on the launch stream)"
    kernel, n_splits, launches = wl.plan()
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
        "data": "synthetic (seeded spectrum-decay weights, Gaussian latents drawn on the device, Gaussian queries)",
        "config": {"workload": name, "batch": cfg.batch, "tokens": cfg.T, "heads": cfg.n_heads,
                   "head_dim": cfg.head_dim, "group_size": cfg.group_size, "rank": cfg.rank,
                   "latent_dtype": cfg.latent_dtype, "mode": cfg.mode, "hadamard": cfg.hadamard,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "flushed (512 MB write) before every timed step",
                   "bytes_per_step": work["decode_bytes"], "flops_per_step": work["flops"],
                   "dense_fp16_kv_bytes_per_step": work["dense_fp16_kv_bytes"], "n_splits": n_splits},
        "dense_equiv_gbs": round(job_throughput_gbs(world, work["dense_fp16_kv_bytes"], ms_per_step), 1),
        "roofline": roof,
        "kernel_us": stats_us(kernel_ms_list),
        "step_us": stats_us(step_ms),
        "kernel_launches_traced": len(kernel_ms_list),
        "e2e": {"value": round(job_throughput_gbs(world, work["decode_bytes"], e2e_step), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_step, 6),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke},
        "gpu_launches": wl.launches_per_step * K,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 4),
    }
    if rank == 0 and not args.no_cpu_baseline:
        sample = wl.oracle_sample()
        result["cpu_baseline"] = cpu_baseline(sample, work, budget_s=args.cpu_seconds)
        result["parity_sample"] = sample.compare(wl.out.cpu().double().numpy())
    headline_entry = per_config_entry(name, cfg, work, step_ms, kernel_ms_list, clk.summary(), wl, peaks, peaks_src,
                                      result.get("cpu_baseline"), result.get("parity_sample"))
    wl.close()
    del wl
    torch.cuda.empty_cache()
    if rank == 0 and world == 1 and not args.no_per_config:
        result["per_config"] = run_per_config(args, dev, flush, name, headline_entry, peaks, peaks_src)
        result["t_sweep"] = run_t_sweep(args, dev, flush, peaks, peaks_src)
        result["next_rows"] = run_next_rows(args, dev, flush, peaks, peaks_src)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return result if rank == 0 else None


def per_config_entry(name, cfg, work, step_ms, kernel_ms, clocks, wl, peaks, peaks_src, cpu=None, parity=None):
    med = pct(kernel_ms, 50)
    roof = roofline_for(cfg, work, med, peaks, peaks_src, long_step=False)
    roof["traffic"] = recorded_traffic(name, wl.kernel_name, cfg)
    roof["duration"] = "median decode-kernel launch"
    kernel, n_splits, launches = wl.plan()
    e = {"batch": cfg.batch, "tokens": cfg.T, "latent_dtype": cfg.latent_dtype, "mode": cfg.mode,
         "kernel": wl.kernel_name, "n_splits": n_splits, "gpu_launches_per_step": 1 + launches,
         "decode_kernel_us": stats_us(kernel_ms), "step_us": stats_us(step_ms),
         "latent_gbs": round(work["decode_bytes"] / (med / 1e3) / 1e9, 1),
         "dense_equiv_gbs": round(work["dense_fp16_kv_bytes"] / (med / 1e3) / 1e9, 1),
         "bytes": work["decode_bytes"], "flops": work["flops"], "roofline": roof, "clocks": clocks}
    if cpu is not None:
        e["cpu_baseline"] = cpu
    if parity is not None:
        e["parity_sample"] = parity
    return e


def run_per_config(args, dev, flush, headline, headline_entry, peaks, peaks_src):
    """Every benchmark workload at its full size, one after the other: 10 warm-up steps, then at
    least 50 timed steps (500 at T <= 4K), L2 flushed before each; median/p10/p90 of the decode
    kernel and of the step, roofline, recorded traffic, clocks and the oracle's CPU baseline."""
    import torch
    out = {}
    for name in PER_CONFIG_ORDER:
        if name == headline:
            out[name] = headline_entry
            continue
        cfg = config_of(name)
        t_gen = time.perf_counter()
        wl = GpuWorkload(cfg, dev)
        gen_s = time.perf_counter() - t_gen
        for _ in range(10):
            flush.zero_()
            wl.step()
        torch.cuda.synchronize()
        n = 500 if cfg.T <= 4096 else max(50, args.per_config_steps)
        step_ms, kms, clocks = timed_steps(wl, n, flush, dev.index)
        work = step_work(cfg)
        cpu = parity = None
        if not args.no_cpu_baseline:
            sample = wl.oracle_sample()
            cpu = cpu_baseline(sample, work, budget_s=args.per_config_cpu_seconds)
            parity = sample.compare(wl.out.cpu().double().numpy())
            if name in SINGLE_CORE_ORACLE:
                cpu["single_core"] = single_core_oracle(sample, work, args.per_config_cpu_seconds)
        e = per_config_entry(name, cfg, work, step_ms, kms, clocks, wl, peaks, peaks_src, cpu, parity)
        e["setup_s"] = round(gen_s, 2)
        out[name] = e
        print(f"[bench] {name}: decode kernel median {e['decode_kernel_us']['median']} us, "
              f"{e['roofline']['bound']} frac {e['roofline']['frac']}", file=sys.stderr, flush=True)
        wl.close()
        del wl
        torch.cuda.empty_cache()
    return out


# T sweep: each 64K workload's decode at T = 4K, 8K, 16K, 32K and 64K (same batch and layer)
T_SWEEP = (4096, 8192, 16384, 32768, 65536)
T_SWEEP_WORKLOADS = ("llama2-7b-rope-int4-hadamard-b4-t64k", "llama2-7b-absorbed-fp16-b4-t64k")


def run_t_sweep(args, dev, flush, peaks, peaks_src):
    """The decode kernel of each T_SWEEP_WORKLOADS workload at every T of T_SWEEP: 5 warm-up steps,
    then 30 timed steps (100 at T <= 8K), L2 flushed before each; median decode kernel, latent and
    dense-equivalent GB/s, and the roofline fraction."""
    import torch
    out = {}
    for name in T_SWEEP_WORKLOADS:
        rows = []
        for T in T_SWEEP:
            cfg = config_of(name, tokens=T)
            wl = GpuWorkload(cfg, dev)
            for _ in range(5):
                flush.zero_()
                wl.step()
            torch.cuda.synchronize()
            _, kms, _ = timed_steps(wl, 100 if T <= 8192 else 30, flush)
            work = step_work(cfg)
            med = pct(kms, 50)
            roof = roofline_for(cfg, work, med, peaks, peaks_src, long_step=False)
            rows.append({"tokens": T, "n_splits": wl.plan()[1], "decode_kernel_us": round(med * 1e3, 2),
                         "latent_gbs": round(work["decode_bytes"] / (med / 1e3) / 1e9, 1),
                         "dense_equiv_gbs": round(work["dense_fp16_kv_bytes"] / (med / 1e3) / 1e9, 1),
                         "bound": roof["bound"], "frac": roof["frac"]})
            wl.close()
            del wl
            torch.cuda.empty_cache()
        out[name] = rows
        print(f"[bench] T sweep {name}: " + ", ".join(f"{r['tokens'] // 1024}K {r['decode_kernel_us']} us "
                                                     f"({r['frac']})" for r in rows), file=sys.stderr, flush=True)
    return out


# ---------------------------------------------------------------------------
# The steps around the decode: output projection (and the rows after it)
# ---------------------------------------------------------------------------

def event_times(fn, n, flush):
    """n CUDA-event timings (ms) of fn() on the current stream, L2 flushed before each."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(n):
        flush.zero_()
        ev[i][0].record()
        fn()
        ev[i][1].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def hbm_roofline(nbytes, ms, peaks, peaks_src):
    ach = nbytes / (ms / 1e3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    return {"bound": "hbm", "achieved": round(ach, 1), "peak": hbm, "unit": "GB/s", "frac": round(ach / hbm, 4),
            "roofline_us": round(nbytes / (hbm * 1e9) * 1e6, 2), "peak_source": f"hbm_gbs of {peaks_src}",
            "duration": "median launch"}


def oracle_seconds(fn, budget_s):
    """(calls, seconds) of the oracle function run repeatedly for about budget_s seconds."""
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or done == 0:
        fn()
        done += 1
    return done, time.perf_counter() - t0


def bench_output_projection(args, dev, flush, peaks, peaks_src, batch):
    """y = o (B_v W_o): the fused-weight GEMV of the Llama-2-7B layer (32 heads, r_v 256, d 4096;
    a 64 MB fp16 weight), o as the decode kernel writes it."""
    import numpy as np
    import torch
    from oracle import palu_oracle as O
    from rank_kv_cache_gb300 import palu as P
    from synthetic import gen
    cfg = gen.ROPE_FP16
    n, r_v, d = cfg.n_heads, cfg.rank, cfg.hidden
    fac, _ = gen.factors(cfg)
    wo = torch.randn((n * cfg.head_dim, d), generator=torch.Generator().manual_seed(7)) / math.sqrt(d)
    proj = P.OutputProjection(gen.storage_round(fac["v"][1], "f16").to(dev), wo.half().to(dev), n_heads=n,
                              head_dim=cfg.head_dim, group_size=cfg.group_size, rank_v=r_v, max_batch=batch)
    o = torch.randn((batch, n * r_v), generator=torch.Generator().manual_seed(8)).to(dev)
    y = torch.empty((batch, d), dtype=torch.float32, device=dev)
    for _ in range(10):
        proj(o, y)
    torch.cuda.synchronize()
    ms = event_times(lambda: proj(o, y), 500, flush)
    nbytes = proj.w.numel() * 2 + o.numel() * 4 + y.numel() * 4
    med = pct(ms, 50)
    e = {"batch": batch, "k_dim": n * r_v, "d_model": d, "w_dtype": "f16", "kernel": "oproj_kernel",
         "gpu_launches_per_step": 1, "kernel_us": stats_us(ms), "bytes": nbytes,
         "roofline": hbm_roofline(nbytes, med, peaks, peaks_src)}
    w64 = proj.w.cpu().double().numpy()
    o64 = o.cpu().double().numpy().reshape(batch, n, r_v)
    ref = O.project_fused(o64, w64)
    e["parity_sample"] = {"max_err_over_max_ref": float(np.abs(y.cpu().double().numpy() - ref).max() /
                                                        np.abs(ref).max())}
    if not args.no_cpu_baseline:
        calls, sec = oracle_seconds(lambda: O.project_fused(o64, w64), 2.0)
        e["cpu_baseline"] = {"value": round(nbytes * calls / sec / 1e9, 4), "unit": "GB/s", "cores": _blas_threads(),
                             "kind": "oracle", "seconds": round(sec, 2),
                             "sample": f"{calls} full projections (float64 NumPy, per-head matvecs)"}
    del proj
    return e


def tensor_roofline(flops, ms, peaks, peaks_src):
    ach = flops / (ms / 1e3) / 1e12
    tc = float(peaks["bf16_tflops"])
    return {"bound": "tensor", "achieved": round(ach, 1), "peak": tc, "unit": "TFLOP/s", "frac": round(ach / tc, 4),
            "roofline_us": round(flops / (tc * 1e12) * 1e6, 2), "peak_source": f"bf16_tflops of {peaks_src}",
            "duration": "median launch"}


def bench_prefill(args, dev, flush, peaks, peaks_src, batch, T, latent_dtype):
    """H = x A for a prefill of batch x T tokens of the Llama-2-7B layer (d 4096, 8 groups, rank 256,
    key and value), written into a cache of latent_dtype; x fp16."""
    import numpy as np
    import torch
    from oracle import palu_oracle as O
    from rank_kv_cache_gb300 import palu as P
    from synthetic import gen
    cfg = gen.ROPE_INT4 if latent_dtype == "int4" else gen.ROPE_FP16
    fac, _ = gen.factors(cfg)
    bk = gen.storage_round(fac["k"][1], "f16").to(dev)
    attn = P.PaluAttention(bk, n_heads=cfg.n_heads, head_dim=cfg.head_dim, group_size=cfg.group_size,
                           rank_k=cfg.rank, rank_v=cfg.rank, latent_dtype=latent_dtype, q_dtype="f16", mode="rope",
                           max_batch=batch, max_tokens=T)
    cache = P.LatentCache(batch, T, cfg.n_groups, cfg.rank, cfg.rank, latent_dtype, device=dev)
    ak = gen.storage_round(fac["k"][0], "f16").to(dev)
    av = gen.storage_round(fac["v"][0], "f16").to(dev)
    w = attn.prepare_down_proj(ak, av, dtype="f16")
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    x = torch.randn((batch, T, cfg.hidden), generator=g, device=dev, dtype=torch.float32).half()
    slot = torch.zeros(batch, dtype=torch.int32, device=dev)
    for _ in range(5):
        attn.project(w, x, cache, slot)
    torch.cuda.synchronize()
    ms = event_times(lambda: attn.project(w, x, cache, slot), 50, flush)
    attn.check_device()
    M, d, N = batch * T, cfg.hidden, 2 * cfg.n_groups * cfg.rank
    flops = 2 * M * d * N
    med = pct(ms, 50)
    e = {"batch": batch, "tokens": T, "d_model": d, "n_out": N, "x_dtype": "f16", "latent_dtype": latent_dtype,
         "kernel": "project_latents_kernel", "gpu_launches_per_step": 1, "kernel_us": stats_us(ms), "flops": flops,
         "roofline": tensor_roofline(flops, med, peaks, peaks_src)}
    # parity sample and oracle baseline: 64 tokens of batch row 0, group 0 of the key side
    xs = x[0, :64].float().cpu().double().numpy()[None]
    a0 = ak[:1].float().cpu().double().numpy()
    ref = O.project_latents(xs, a0)[0, :, 0, :]
    if latent_dtype == "int4":
        codes, sc = O.quantize_int4(ref.astype(np.float32))
        got = O.dequant_int4(cache.hk[0, :64, 0].cpu().numpy(), cache.k_scale[0, :64, 0].cpu().numpy())
        e["parity_sample"] = {"tokens": 64, "max_abs_err_vs_oracle_dequant": float(np.abs(got - O.dequant_int4(
            O.pack_int4(codes), sc)).max()), "scale_units_max": float(np.abs(got - ref).max() / float(sc.max()))}
    else:
        got = cache.hk[0, :64, 0].float().cpu().double().numpy()
        e["parity_sample"] = {"tokens": 64, "max_err_over_max_ref": float(np.abs(got - ref).max() / np.abs(ref).max())}
    if not args.no_cpu_baseline:
        a_all = ak.float().cpu().double().numpy()
        calls, sec = oracle_seconds(lambda: O.project_latents(xs, a_all), 2.0)
        toks = 64 * calls
        e["cpu_baseline"] = {"value": round(2 * toks * d * (N // 2) / sec / 1e12, 6), "unit": "TFLOP/s",
                             "cores": _blas_threads(), "kind": "oracle", "seconds": round(sec, 2),
                             "sample": f"{calls} x 64 tokens of the key side (float64 NumPy)"}
    attn.close()
    return e


def bench_hybrid(args, dev, flush, peaks, peaks_src, sinks=4, window=64):
    """Decode over a hybrid cache: the Llama-2-7B int4 layer at batch 4 with `sinks` + `window`
    dense fp16 tokens around a latent middle of 65536 - sinks - window tokens (positions
    sinks .. sinks + T_mid - 1, the query at 65535). Times the whole call (latent decode + dense
    merge) and, from the library's trace, the latent decode kernel alone."""
    import torch
    from rank_kv_cache_gb300 import palu as P
    from synthetic import gen
    cfg = gen.ROPE_INT4.with_(T=gen.ROPE_INT4.T - sinks - window)
    wl = GpuWorkload(cfg, dev, max_position=gen.ROPE_INT4.T)
    B, T, n, d_h = cfg.batch, cfg.T, cfg.n_heads, cfg.head_dim
    D = sinks + window
    g = torch.Generator(device=dev)
    g.manual_seed(13)
    dk = torch.randn((B, D, n, d_h), generator=g, device=dev).half()
    dv = torch.randn((B, D, n, d_h), generator=g, device=dev).half()
    nd = torch.full((B,), D, dtype=torch.int32, device=dev)
    pos = (torch.arange(T, dtype=torch.int32, device=dev) + sinks).repeat(B, 1).contiguous()
    qp = torch.full((B,), sinks + T + window - 1, dtype=torch.int32, device=dev)
    seq = torch.full((B,), T, dtype=torch.int32, device=dev)
    out = torch.empty((B, n, cfg.rank), dtype=torch.float32, device=dev)
    od = torch.empty((B, n, d_h), dtype=torch.float32, device=dev)
    lse = torch.empty((B, n), dtype=torch.float32, device=dev)

    def call():
        wl.attn.decode_hybrid(wl.q, wl.cache, seq, dk, dv, nd, max_seq_len=T, positions=pos, q_pos=qp, out=out,
                              out_dense=od, lse=lse)

    for _ in range(5):
        call()
    torch.cuda.synchronize()
    P.check(P.palu_attn_trace_enable(wl.attn.handle, 1))
    ms = event_times(call, 50, flush)
    st, kms = P.palu_attn_trace_times(wl.attn.handle)
    P.check(st)
    P.check(P.palu_attn_trace_enable(wl.attn.handle, 0))
    wl.attn.check_device()
    work = step_work(cfg)
    dense_bytes = 2 * B * D * n * d_h * 2
    e = {"batch": B, "sink_tokens": sinks, "window_tokens": window, "latent_tokens": T, "latent_dtype": "int4",
         "dense_dtype": "f16", "kernels": ["decode_tc_kernel", "merge_dense_kernel"], "gpu_launches_per_step": 2,
         "call_us": stats_us(ms), "latent_decode_kernel_us": stats_us(kms),
         "dense_merge_us_median": round((pct(ms, 50) - pct(kms, 50)) * 1e3, 2),
         "bytes": work["decode_bytes"] + dense_bytes, "flops": work["flops"],
         "roofline": roofline_for(cfg, work, pct(ms, 50), peaks, peaks_src, long_step=False)}
    e["roofline"]["duration"] = "median whole call (latent decode + dense merge)"
    wl.close()
    return e


def bench_paged(args, dev, flush, peaks, peaks_src, sinks=4, window=64, page=32, rank=16):
    """Decode over a page-factorised cache (PuzzleKV section 3.3) at the Llama-2-7B shape: batch 4,
    32 heads, d_h 128, 64K tokens as `sinks` + `window` dense fp16 tokens and the rest in pages of 32
    tokens stored as rank-16 fp16 factors (10 KB per page and head). Times the whole call (the paged
    kernel and the dense merge); bound by HBM."""
    import numpy as np
    import torch
    from oracle import palu_oracle as O
    from rank_kv_cache_gb300 import palu as P
    B, n, d_h, T = 4, 32, 128, 65536
    D = sinks + window
    n_pages = (T - D) // page
    bk = torch.zeros((8, 256, 4 * d_h), dtype=torch.float16, device=dev)
    attn = P.PaluAttention(bk, n_heads=n, head_dim=d_h, group_size=4, rank_k=256, rank_v=256, latent_dtype="f16",
                           q_dtype="f16", mode="rope", max_batch=B, max_tokens=T, max_position=T)
    g = torch.Generator(device=dev)
    g.manual_seed(17)
    rec = (torch.randn((B, n_pages, n, 320 * rank), generator=g, device=dev) * 0.2).half()
    dk = torch.randn((B, D, n, d_h), generator=g, device=dev).half()
    dv = torch.randn((B, D, n, d_h), generator=g, device=dev).half()
    q = torch.randn((B, n, d_h), generator=g, device=dev).half()
    npg = torch.full((B,), n_pages, dtype=torch.int32, device=dev)
    nd = torch.full((B,), D, dtype=torch.int32, device=dev)
    qp = torch.full((B,), T - 1, dtype=torch.int32, device=dev)
    out = torch.empty((B, n, d_h), dtype=torch.float32, device=dev)
    od = torch.empty((B, n, d_h), dtype=torch.float32, device=dev)
    lse = torch.empty((B, n), dtype=torch.float32, device=dev)

    def call():
        attn.decode_paged(q, rec, npg, max_pages=n_pages, q_pos=qp, dense_k=dk, dense_v=dv, dense_n=nd, out=out,
                          out_dense=od, lse=lse)

    for _ in range(5):
        call()
    torch.cuda.synchronize()
    ms = event_times(call, 50, flush)
    attn.check_device()
    nbytes = rec.numel() * 2 + 2 * dk.numel() * 2
    med = pct(ms, 50)
    e = {"batch": B, "n_heads": n, "page_tokens": page, "rank": rank, "pages_per_row": n_pages,
         "sink_tokens": sinks, "window_tokens": window, "dtype": "f16",
         "kernels": ["paged_decode_kernel", "merge_dense_kernel"], "gpu_launches_per_step": 2,
         "call_us": stats_us(ms), "bytes": nbytes, "roofline": hbm_roofline(nbytes, med, peaks, peaks_src)}
    e["roofline"]["duration"] = "median whole call (paged decode + dense merge)"
    # the oracle on one (row, head), against the same inputs
    b1, h1 = 1, 7
    r64 = rec[b1, :, h1].float().cpu().double().numpy()
    o1, o2, o3 = page * rank, page * rank + rank * d_h, 2 * page * rank + rank * d_h
    fk = (r64[:, :o1].reshape(1, n_pages, 1, page, rank), r64[:, o1:o2].reshape(1, n_pages, 1, rank, d_h),
          r64[:, o2:o3].reshape(1, n_pages, 1, page, rank), r64[:, o3:].reshape(1, n_pages, 1, rank, d_h))
    args64 = (q[b1:b1 + 1, h1:h1 + 1].cpu().double().numpy(), *fk, [n_pages],
              dk[b1:b1 + 1, :, h1:h1 + 1].cpu().double().numpy(), dv[b1:b1 + 1, :, h1:h1 + 1].cpu().double().numpy(),
              [D])
    ref_p, ref_d, ref_lse = O.decode_paged(*args64, mode="rope", q_pos=[T - 1])
    got = (out[b1, h1] + od[b1, h1]).cpu().double().numpy()
    ref = ref_p[0, 0] + ref_d[0, 0]
    e["parity_sample"] = {"heads": [[b1, h1]], "max_err_over_max_ref": float(np.abs(got - ref).max() / np.abs(ref).max()),
                          "lse_abs_err": float(abs(lse[b1, h1].item() - ref_lse[0, 0]))}
    if not args.no_cpu_baseline:
        calls, sec = oracle_seconds(lambda: O.decode_paged(*args64, mode="rope", q_pos=[T - 1]), 2.0)
        per_head = nbytes / (B * n)
        e["cpu_baseline"] = {"value": round(per_head * calls / sec / 1e9, 4), "unit": "GB/s",
                             "cores": _blas_threads(), "kind": "oracle", "seconds": round(sec, 2),
                             "sample": f"{calls} decodes of one (row, head) over its {n_pages} pages and {D} dense "
                                       "tokens (float64 NumPy)"}
    attn.close()
    del rec
    torch.cuda.empty_cache()
    return e


VARIANTS = (
    # name, workload base, overrides, descriptor flags
    ("llama2-7b-rope-fp16k-int4v-b4-t64k", "ROPE_FP16", dict(batch=4, T=65536, v_dtype="int4"), 0),
    ("llama2-7b-absorbed-alibi-fp16-b4-t64k", "ABSORBED_FP16", dict(), 1),
    ("llama2-7b-rope-fp16-mlrd-s1-r64-b1-t4k", "ROPE_FP16", dict(group_size=1, rank=64), 0),
    ("llama2-7b-rope-fp16-glrd-s2-r256-b1-t4k", "ROPE_FP16", dict(group_size=2), 0),
    ("llama2-7b-rope-fp16-glrd-s4-r256-b1-t4k", "ROPE_FP16", dict(), 0),
    ("llama2-7b-rope-fp16-glrd-s8-r256-b1-t4k", "ROPE_FP16", dict(group_size=8), 0),
    ("llama2-7b-rope-fp16-jlrd-s32-r256-b1-t4k", "ROPE_FP16", dict(group_size=32), 0),
    ("llama2-7b-absorbed-fp16-glrd-s8-b4-t64k", "ABSORBED_FP16", dict(group_size=8), 0),
    ("llama2-7b-absorbed-fp16-jlrd-s32-b4-t64k", "ABSORBED_FP16", dict(group_size=32), 0),
)


def bench_variant(args, dev, flush, peaks, peaks_src, base, over, flags):
    """One decode variant at full size: append + decode steps, L2 flushed before each, the decode
    kernel timed from the library's trace."""
    import torch
    from synthetic import gen
    cfg = getattr(gen, base).with_(**over)
    wl = GpuWorkload(cfg, dev, flags=flags)
    for _ in range(5):
        flush.zero_()
        wl.step()
    torch.cuda.synchronize()
    step_ms, kms, clocks = timed_steps(wl, 50 if cfg.T > 4096 else 200, flush, dev.index)
    work = step_work(cfg)
    e = per_config_entry(f"variant:{base}", cfg, work, step_ms, kms, clocks, wl, peaks, peaks_src)
    e.update({"group_size": cfg.group_size, "rank": cfg.rank, "value_dtype": cfg.value_dtype,
              "alibi": bool(flags & 1), "rebuild_flops_per_token": work["flops"] // (cfg.batch * cfg.T)})
    wl.close()
    return e


def next_row_table():
    """name -> function(args, dev, flush, peaks, peaks_src) of every measurement next to the decode
    workloads, in the order the bench line lists them."""
    t = {}
    for b in (1, 4):
        t[f"llama2-7b-oproj-fp16-b{b}"] = (lambda b: lambda *a: bench_output_projection(*a, b))(b)
    for name, base, over, flags in VARIANTS:
        t[name] = (lambda base, over, flags: lambda *a: bench_variant(*a, base, over, flags))(base, over, flags)
    t["llama2-7b-hybrid-int4-b4-t64k-s4-w64"] = lambda *a: bench_hybrid(*a)
    t["puzzlekv-paged-fp16-b4-t64k-p32-r16-s4-w64"] = lambda *a: bench_paged(*a)
    for b, T, lat in ((1, 4096, "int4"), (4, 4096, "f16")):
        t[f"llama2-7b-prefill-{lat}-b{b}-t4k"] = (lambda b, T, lat: lambda *a: bench_prefill(*a, b, T, lat))(b, T, lat)
    return t


def run_next_rows(args, dev, flush, peaks, peaks_src, only=None):
    """The steps next to the decode kernel (output projection, granularity and storage variants,
    hybrid cache, prefill producer), each timed with CUDA events (L2 flushed before each launch)
    against its own roofline; `only` restricts the run to one of them."""
    import torch
    out = {}
    for name, fn in next_row_table().items():
        if only is not None and name != only:
            continue
        out[name] = e = fn(args, dev, flush, peaks, peaks_src)
        t = e.get("kernel_us") or e.get("decode_kernel_us") or e.get("call_us")
        print(f"[bench] {name}: median {t['median']} us, {e['roofline']['bound']} frac {e['roofline']['frac']}",
              file=sys.stderr, flush=True)
        torch.cuda.empty_cache()
    return out


def run_one_next_row(args):
    """--next-row NAME: that measurement alone, printed as one JSON line (profiling runs)."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    peaks, peaks_src = load_peaks()
    return {"next_row": run_next_rows(args, dev, flush, peaks, peaks_src, only=args.next_row)}


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
    """The oracle on one G-LRD group (batch row 0, group 0) of the workload: the s heads that read
    it, over all T tokens, on storage-rounded inputs (int4: the oracle's own quantisation)."""

    def __init__(self, cfg, hk, hv, q, bk):
        import numpy as np
        from oracle import palu_oracle as O
        from synthetic import gen
        self.O, self.np, self.cfg = O, np, cfg
        if cfg.latent_dtype == "int4":
            ck, sk = O.quantize_int4(hk)
            cv, sv = O.quantize_int4(hv)
            hk = O.dequant_int4(O.pack_int4(ck), sk)
            hv = O.dequant_int4(O.pack_int4(cv), sv)
        else:
            hk = gen.storage_round(hk, cfg.latent_dtype).double().numpy()
            hv = gen.storage_round(hv, cfg.latent_dtype).double().numpy()
        s = cfg.group_size
        self.hk = np.ascontiguousarray(hk[None, :, None, :])    # [1][T][1][r]
        self.hv = np.ascontiguousarray(hv[None, :, None, :])
        self.q = gen.storage_round(q[:1, :s], cfg.q_dtype).double().numpy()
        self.bk = bk.double().numpy()[:1]                        # storage-rounded torch tensor
        self.seq = np.array([cfg.T])
        self.heads = [(0, j) for j in range(s)]
        self.results = {}

    def run(self, head):
        c = self.cfg
        o, lse = self.O.decode(self.q, self.hk, self.hv, self.bk, self.seq, c.group_size, mode=c.mode,
                               theta=c.theta, heads=[head])
        self.results[head] = (o[head], lse[head])

    def compare(self, gpu_out):
        """max |GPU - oracle| over the heads the oracle has computed (batch row 0, group 0)."""
        if not self.results:
            return None
        d = max(float(self.np.abs(gpu_out[0, j] - o).max()) for (_, j), (o, _) in self.results.items())
        ref = max(float(self.np.abs(o).max()) for o, _ in self.results.values())
        return {"heads": len(self.results), "max_abs_err": d, "max_err_over_max_ref": d / ref if ref else d}


def cpu_baseline(sample, work, budget_s=12.0):
    """Time the oracle as it stands on this host's cores over a bounded sample of the workload."""
    cfg = sample.cfg
    total_heads = cfg.batch * cfg.n_heads
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or done == 0:
        sample.run(sample.heads[done % len(sample.heads)])
        done += 1
    el = time.perf_counter() - t0
    frac = done / total_heads
    return {"value": round(work["decode_bytes"] * frac / el / 1e9, 4), "unit": "GB/s", "cores": _blas_threads(),
            "kind": "oracle", "seconds": round(el, 2),
            "sample": f"{done} single-head decodes (the {len(sample.heads)} heads of batch row 0, group 0, "
                      f"cycled) of the workload's {total_heads}, all {cfg.T} tokens each, float64 NumPy"}


def single_core_oracle(sample, work, budget_s):
    """The same oracle sample on one core: a child process pinned to one CPU with BLAS threads
    set to 1 before NumPy loads."""
    import numpy as np
    cfg = sample.cfg
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "sample.npz")
        np.savez(path, q=sample.q, hk=sample.hk, hv=sample.hv, bk=sample.bk, seq=sample.seq)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        cmd = [sys.executable, os.path.abspath(__file__), "--oracle-child", path, "--oracle-child-cfg",
               json.dumps({"group_size": cfg.group_size, "mode": cfg.mode, "theta": cfg.theta}),
               "--cpu-seconds", str(budget_s)]
        res = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=budget_s * 10 + 120)
        if res.returncode != 0:
            return {"error": res.stderr.strip().splitlines()[-1:] or ["child failed"]}
        child = json.loads(res.stdout.strip().splitlines()[-1])
    frac = child["heads"] / (cfg.batch * cfg.n_heads)
    return {"value": round(work["decode_bytes"] * frac / child["seconds"] / 1e9, 4), "unit": "GB/s", "cores": 1,
            "ms_per_head": round(child["seconds"] / child["heads"] * 1e3, 2),
            "ms_per_step_equivalent": round(child["seconds"] / frac * 1e3, 1), "kind": "oracle"}


def oracle_child(path, cfg_json, budget_s):
    os.sched_setaffinity(0, {sorted(os.sched_getaffinity(0))[0]})
    import numpy as np
    from oracle import palu_oracle as O
    c = json.loads(cfg_json)
    z = np.load(path)
    heads = [(0, j) for j in range(z["q"].shape[1])]
    done = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < budget_s or done == 0:
        O.decode(z["q"], z["hk"], z["hv"], z["bk"], z["seq"], c["group_size"], mode=c["mode"], theta=c["theta"],
                 heads=[heads[done % len(heads)]])
        done += 1
    print(json.dumps({"heads": done, "seconds": time.perf_counter() - t0}))


def run_reference(args, cfg, name):
    world, rank, _ = _dist()
    if rank != 0:
        return None
    import numpy as np
    from synthetic import gen
    work = step_work(cfg)
    fac, _ = gen.factors(cfg)
    sample = OracleSample(cfg, gen.sample_group_latents(cfg, "k"), gen.sample_group_latents(cfg, "v"),
                          gen.draw_query(cfg), gen.storage_round(fac["k"][1], cfg.bk_dtype))
    # one head per step over all T tokens, cycling through the heads of batch row 0, group 0
    frac = 1 / (cfg.batch * cfg.n_heads)
    for i in range(args.warmup):
        sample.run(sample.heads[i % len(sample.heads)])
    t0 = time.perf_counter()
    for i in range(args.steps):
        sample.run(sample.heads[i % len(sample.heads)])
    el = time.perf_counter() - t0
    ms = el / args.steps * 1e3
    val = round(work["decode_bytes"] * frac / (ms / 1e3) / 1e9, 4)
    desc = (f"one head per step (cycling over the {len(sample.heads)} heads of batch row 0, group 0) of the "
            f"workload's {cfg.batch * cfg.n_heads}, all {cfg.T} tokens, float64 NumPy")
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
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--per-config-steps", type=int, default=100, help="timed steps per workload above T=4K")
    ap.add_argument("--per-config-cpu-seconds", type=float, default=3.0)
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (profiling runs)")
    ap.add_argument("--tokens", type=int, default=None, help="override the workload's T (profiling runs)")
    ap.add_argument("--next-row", default=None, help="run one next-row measurement alone (profiling runs)")
    ap.add_argument("--oracle-child", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-child-cfg", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.oracle_child:
        oracle_child(args.oracle_child, args.oracle_child_cfg, args.cpu_seconds)
        return
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.next_row is not None:
        if args.next_row not in next_row_table():
            ap.error(f"--next-row must be one of {sorted(next_row_table())}")
        print(json.dumps(run_one_next_row(args)), flush=True)
        return
    cfg = config_of(args.workload, args.batch, args.tokens)
    res = run_reference(args, cfg, args.workload) if args.impl == "reference" else run_gpu(args, cfg, args.workload)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()

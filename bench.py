#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path on GB300.

One step = one prefill pass and one split-KV decode pass, each through the C ABI, on synthetic
inputs of the pages' shapes already resident in device memory:
  prefill: grouped-query causal prefill, B=1, Hq=64, Hkv=8, N=8192, d=128, bf16
           (the 70B-class head shape), FLOPs counted as 4*B*Hq*N^2*d/2 (causal);
  decode:  B=64 sequences, Hq=64, Hkv=8, d=128, bf16, lengths ~ U[1024, 32768] (seed 5000),
           512-token splits, algorithmic bytes = K + V + q + o + lse.
The headline ``value`` is prefill TFLOP/s (whole job: all ranks' FLOPs / the slowest rank's
prefill time); decode GB/s is reported beside it under ``decode``.  Kernel durations come from
CUDA events on the launching stream.  Both workloads are larger than L2 (302 MB and 4.4 GB), so
no L2 flush is inserted between steps.

``--impl reference`` times the fp64 CPU oracle (the reference definition) on a bounded sample of
the same prefill workload, on this machine's host cores.

Multi-GPU (torchrun): every rank runs the same workload on its own GPU (replicas, weak scaling);
there is no collective on the data path.  A barrier and a max-over-ranks reduction frame the
timed region.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "attn fwd TFLOP/s & % BF16 tensor peak; decode KV-read GB/s & % HBM peak"


# ----------------------------------------------------------------------------------------
# distributed helpers (also used by the CPU gloo test)
# ----------------------------------------------------------------------------------------
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(values, device=None):
    """Element-wise max over ranks of a list of floats (identity without a process group)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def aggregate(units_per_rank: float, seconds_per_rank: float, world: int, device=None) -> float:
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    (t_max,) = reduce_max([seconds_per_rank], device)
    return units_per_rank * world / t_max


def barrier(device=None):
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized():
        if device is not None and str(device).startswith("cuda"):
            dist.barrier(device_ids=[int(str(device).split(":")[1])])
        else:
            dist.barrier()


# ----------------------------------------------------------------------------------------
# peaks, clocks, profiles
# ----------------------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == "start":
            self.t_start = time.time()
        else:
            self.t_stop = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(2 * self.period / 1000.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sel = [l for t, l in self.lines if self.t_start is None or
               (self.t_start - 0.06 <= t <= (self.t_stop or t) + 0.06)]
        if not sel:
            sel = [l for _, l in self.lines]
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in sel:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {
            "sm_mhz": float(np.median(sm)) if sm else None,
            "sm_max_mhz": float(max(smax)) if smax else None,
            "power_w_max": float(max(power)) if power else None,
            "samples": len(sm),
            "reasons": sorted(reasons),
        }


def source_sha(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, sources):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel]
        if e.get("source_sha") != source_sha(sources):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


FWD_SOURCES = ["exact_io_aware_09_gb300/csrc/attn_fwd.cu", "exact_io_aware_09_gb300/csrc/ptx.cuh",
               "exact_io_aware_09_gb300/csrc/internal.h"]
DEC_SOURCES = ["exact_io_aware_09_gb300/csrc/attn_decode.cu", "exact_io_aware_09_gb300/csrc/ptx.cuh",
               "exact_io_aware_09_gb300/csrc/internal.h"]


# ----------------------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample
# ----------------------------------------------------------------------------------------
def prefill_sample_rows(cfg, n_rows, seed=0):
    rng = np.random.default_rng(seed)
    n = cfg.B * cfg.Hq * cfg.N_q
    return np.sort(rng.choice(n, size=n_rows, replace=False)).astype(np.int64)


def row_flops(cfg, rows):
    """Exact FLOPs of the selected rows: 4*d per visible key (2 for Q K^T, 2 for P V)."""
    i = rows % cfg.N_q
    vis = np.minimum(i + (cfg.N_kv - cfg.N_q) + 1, cfg.N_kv) if cfg.causal else np.full_like(i, cfg.N_kv)
    return float(4.0 * cfg.d * np.clip(vis, 0, None).sum())


def visible_keys_window(N_q, N_kv, W):
    """Visible keys per query row under the sliding window (bottom-right aligned)."""
    i = np.arange(N_q, dtype=np.int64)
    hi = np.minimum(i + N_kv - N_q, N_kv - 1)
    lo = np.maximum(i + N_kv - N_q - W, 0)
    return np.clip(hi - lo + 1, 0, None)


def visible_keys_blocks(N_q, N_kv, mask, causal, bs=128):
    """Visible keys per query row under a block pattern (and the causal rule if set)."""
    out = np.zeros(N_q, dtype=np.int64)
    keys = np.arange(N_kv, dtype=np.int64)
    for i in range(N_q):
        vis = mask[i // bs][keys // bs] != 0
        if causal:
            vis &= keys <= i + N_kv - N_q
        out[i] = int(vis.sum())
    return out


def time_oracle_prefill(cfg, q, k, v, budget_s=12.0, rows_per_batch=1024, seed=0):
    """The oracle's throughput on random rows of the workload, in batches of rows_per_batch rows
    per call (large enough that its fixed cost per call, about 75 ms, stays a small part)."""
    import oracle

    rng_seed = seed
    done_flops, t_total, n_rows = 0.0, 0.0, 0
    while t_total < budget_s:
        rows = prefill_sample_rows(cfg, rows_per_batch, rng_seed)
        rng_seed += 1
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, cfg.dtype, cfg.B, cfg.Hq, cfg.Hkv, cfg.N_q, cfg.N_kv,
                              cfg.d, cfg.causal, cfg.scale, rows)
        t_total += time.perf_counter() - t0
        done_flops += row_flops(cfg, rows)
        n_rows += len(rows)
    return done_flops / t_total / 1e12, n_rows, t_total


# ----------------------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    import exact_io_aware_09_gb300 as attn
    import synthetic as syn

    rank, world, local = dist_env()
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device(device))
    peaks, peak_src = load_peaks()

    pcfg = syn.CONFIG4
    if args.prefill_heads != pcfg.Hq:
        group = pcfg.Hq // pcfg.Hkv
        if args.prefill_heads <= 0 or args.prefill_heads % group:
            raise SystemExit(f"--prefill-heads must be a positive multiple of {group}")
        pcfg = dataclasses.replace(pcfg, name=f"{pcfg.name}_hq{args.prefill_heads}",
                                   Hq=args.prefill_heads, Hkv=args.prefill_heads // group)
    dcfg = syn.CONFIG5
    if args.decode_batch != dcfg.B:
        lens = tuple(int(x) for x in dcfg.lengths()[: args.decode_batch])
        dcfg = syn.DecodeConfig(f"{dcfg.name}_first{args.decode_batch}", args.decode_batch, dcfg.Hq,
                                dcfg.Hkv, dcfg.d, dcfg.dtype, dcfg.seed, lengths_override=lens)
    do_pre = args.only in ("both", "prefill")
    do_dec = args.only in ("both", "decode")
    # each path's tensors only when it runs (a one-path run, e.g. under a profiler, then holds
    # only its own inputs)
    q = k = v = o = lse = None
    if do_pre:
        q, k, v = pcfg.device_inputs(device)
        o = torch.empty_like(q)
        lse = torch.empty((pcfg.B, pcfg.Hq, pcfg.N_q), device=device, dtype=torch.float32)
    lengths = dcfg.lengths()
    max_len = int(lengths.max())
    cu = dq = dk = dv = do = dl = ws = None
    if do_dec:
        cu = torch.from_numpy(syn.cu_seqlens(lengths)).to(device)
        dq, dk, dv = dcfg.device_inputs(device)
        do = torch.empty_like(dq)
        dl = torch.empty((dcfg.B, dcfg.Hq), device=device, dtype=torch.float32)
        ws = torch.empty(attn.attn_decode_workspace_bytes(dcfg.B, dcfg.Hq, max_len, dcfg.split,
                                                          dcfg.d),
                         device=device, dtype=torch.uint8)
    stream = torch.cuda.current_stream()

    def prefill():
        if do_pre:
            attn.attn_fwd(q, k, v, o=o, lse=lse, causal=True, scale=pcfg.scale, stream=stream)

    def decode():
        if do_dec:
            attn.attn_decode_splitkv(dq, dk, dv, cu, max_len, o=do, lse=dl, split_size=dcfg.split,
                                     scale=dcfg.scale, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        prefill()
        decode()
    torch.cuda.synchronize()
    st = attn.attn_poll_status()
    if st != 0:
        raise SystemExit(f"device status after warm-up: {attn.attn_status_string(st)}")

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    barrier(device)
    torch.cuda.synchronize()
    sampler.mark("start")
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        ev[i][0].record(stream)
        prefill()
        ev[i][1].record(stream)
        decode()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    barrier(device)
    sampler.mark("stop")
    clocks = sampler.stop()
    st = attn.attn_poll_status()
    if st != 0:
        raise SystemExit(f"device status after timing: {attn.attn_status_string(st)}")
    pre_ms = float(sum(e[0].elapsed_time(e[1]) for e in ev))
    dec_ms = float(sum(e[1].elapsed_time(e[2]) for e in ev))
    step_ms = float(ev[0][0].elapsed_time(ev[-1][2]))
    pre_ms_max, dec_ms_max, step_ms_max, wall_max = reduce_max([pre_ms, dec_ms, step_ms, t_wall], device)

    flops = pcfg.flops()
    kv_bytes = dcfg.kv_bytes()
    # K and V read, q read and o written (2 B each), LSE written (4 B)
    dec_bytes = kv_bytes + 2 * (dcfg.B * dcfg.Hq * dcfg.d) * 2 + dcfg.B * dcfg.Hq * 4
    tiny = 1e-9
    value = flops * args.steps * world / (max(pre_ms_max, tiny) / 1e3) / 1e12 if do_pre else None
    dec_gbs = dec_bytes * args.steps * world / (max(dec_ms_max, tiny) / 1e3) / 1e9 if do_dec else None
    # per-launch rooflines of this rank's kernels
    pre_launch_s = max(pre_ms, tiny) / args.steps / 1e3
    dec_launch_s = max(dec_ms, tiny) / args.steps / 1e3
    ach_t = flops / pre_launch_s / 1e12 if do_pre else 0.0
    ach_b = dec_bytes / dec_launch_s / 1e9 if do_dec else 0.0

    # end to end through the public API with host buffers: H2D inputs, call, D2H result
    e2e = run_e2e(args, attn, pcfg, q, k, v, stream, device, world) if (do_pre and not args.no_e2e) else None
    dec_e2e = (run_e2e_decode(args, attn, dcfg, dq, dk, dv, cu, max_len, ws, dec_bytes, stream,
                              device, world) if (do_dec and not args.no_e2e) else None)

    variants = None
    if do_pre and not args.no_variants:
        variants = measure_variants(args, attn, pcfg, q, k, v, o, lse, stream, peaks, peak_src)
    if do_dec and not args.no_variants:
        variants = variants or {}
        variants["decode_paged"] = measure_paged(args, attn, syn, dcfg, dq, dk, dv, do, dl, ws,
                                                 lengths, max_len, dec_bytes, stream, peaks,
                                                 peak_src)

    configs = None
    if args.only in ("both", "configs") and not args.no_configs:
        configs = measure_configs(args, attn, syn, peaks, peak_src, device, stream,
                                  only=args.config)

    cpu = None
    if rank == 0 and world == 1 and do_pre and not args.no_cpu_baseline:
        cpu = cpu_baseline_prefill(pcfg, q, k, v)

    line = {
        "metric": METRIC,
        "value": round(value, 2) if value is not None else None,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms_max / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), drawn on device)",
        "config": {
            "workload": "gqa causal prefill B=1 Hq=64 Hkv=8 N=8192 d=128 bf16 + split-KV decode "
                        "B=64 Hq=64 Hkv=8 d=128 bf16 L~U[1024,32768] split=512",
            "prefill": pcfg.name, "decode": dcfg.name,
            "prefill_flops_per_step": flops, "decode_bytes_per_step": dec_bytes,
            "l2": "no flush: inputs larger than L2 (prefill 302 MB, decode 4.43 GB per step)",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "kernel": "attn_fwd_kernel<128,bf16>",
            "bound": "tensor",
            "achieved": round(ach_t, 2),
            "peak": peaks["bf16_tflops"],
            "peak_source": f"{peak_src} bf16 burst (cuBLAS)",
            "unit": "TFLOP/s",
            "frac": round(ach_t / peaks["bf16_tflops"], 4),
            "frac_of_spec_2250": round(ach_t / 2250.0, 4),
            "traffic": profiled_traffic("attn_fwd_kernel", FWD_SOURCES),
            # compulsory bytes of one launch: Q, K, V read, O written (2 B each), LSE (4 B)
            "algorithmic_bytes": int((2 * pcfg.B * pcfg.Hq * pcfg.N_q * pcfg.d
                                      + 2 * pcfg.B * pcfg.Hkv * pcfg.N_kv * pcfg.d) * 2
                                     + pcfg.B * pcfg.Hq * pcfg.N_q * 4),
        },
        "decode": {
            "value": round(dec_gbs, 1) if dec_gbs is not None else None,
            "unit": "GB/s",
            "ms_per_launch": round(dec_ms / args.steps, 4),
            "roofline": {
                "kernel": "attn_decode_split_kernel + attn_decode_merge_kernel",
                "bound": "hbm",
                "achieved": round(ach_b, 1),
                "peak": peaks["hbm_gbs"],
                "peak_source": f"{peak_src} HBM copy",
                "unit": "GB/s",
                "frac": round(ach_b / peaks["hbm_gbs"], 4),
                "frac_of_spec_8000": round(ach_b / 8000.0, 4),
                "traffic": profiled_traffic("attn_decode_split_kernel", DEC_SOURCES),
            },
            "e2e": dec_e2e,
        },
        "prefill_ms_per_launch": round(pre_ms / args.steps, 4),
        "configs": configs,
        "variants": variants,
        "e2e": e2e,
        "gpu_launches": (int(do_pre) + 2 * int(do_dec)) * args.steps,
        "clocks": clocks,
        "wall_s_timed": round(wall_max, 4),
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


L2_FLUSH_BYTES = 256 << 20   # twice the 129 MB L2


def causal_pairs(N_q, N_kv):
    """Visible (query, key) pairs of one causal head (bottom-right aligned)."""
    i = np.arange(N_q, dtype=np.int64)
    return int(np.clip(np.minimum(i + N_kv - N_q + 1, N_kv), 0, None).sum())


def measure_configs(args, attn, syn, peaks, peak_src, device, stream, only=None):
    """The prefill workloads of the pages' shapes besides the headline one: the single head
    (N=256, d=64, fp16), the GPT-2 shape (B=8, H=12, N=1024, d=64, bf16, causal), the long
    prefill (B=4, H=32, N=4096, d=128, fp16, full and causal) and its x8-logit stress.

    Workloads whose inputs fit in L2 (the single head, the GPT-2 shape) are timed one launch
    at a time with CUDA events on the launching stream, each after a write of a 256 MB buffer
    (twice L2) so that no launch finds its inputs in L2; the others (537 MB of inputs) are
    timed over back-to-back launches, as the headline prefill.  3 warm-up launches.
    TFLOP/s by the pages' convention (4*B*H*N^2*d, halved for causal) and by the exact count of
    visible (query, key) pairs (4*d each); roofline against the measured bf16 dense peak (fp16
    has the same nominal tensor rate)."""
    import torch

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    out = {}
    configs = [syn.CONFIG1, syn.CONFIG2, syn.CONFIG3A, syn.CONFIG3B, syn.CONFIG3SA, syn.CONFIG3SB]
    n_launch = max(10, min(args.steps, 50))
    for cfg in configs:
        if only is not None and cfg.name != only:
            continue
        q, k, v = cfg.device_inputs(device)
        o = torch.empty_like(q)
        lse = torch.empty((cfg.B, cfg.Hq, cfg.N_q), device=device, dtype=torch.float32)
        fn = lambda: attn.attn_fwd(q, k, v, o=o, lse=lse, causal=cfg.causal, scale=cfg.scale,
                                   stream=stream)
        for _ in range(3):
            fn()
        in_bytes = (q.numel() + k.numel() + v.numel()) * q.element_size()
        flushed = in_bytes < L2_FLUSH_BYTES // 2
        torch.cuda.synchronize()
        if flushed:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(n_launch)]
            with torch.cuda.stream(stream):
                for e0, e1 in ev:
                    flush.fill_(1)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
            torch.cuda.synchronize()
            times = sorted(e0.elapsed_time(e1) for e0, e1 in ev)
        else:
            times = []
            for _ in range(3):  # three rounds of back-to-back launches
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(n_launch):
                    fn()
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) / n_launch)
            times.sort()
        st = attn.attn_poll_status()
        if st != 0:
            raise SystemExit(f"device status after {cfg.name}: {attn.attn_status_string(st)}")
        ms = float(np.mean(times))
        pairs = (causal_pairs(cfg.N_q, cfg.N_kv) if cfg.causal else cfg.N_q * cfg.N_kv)
        exact = 4.0 * cfg.d * pairs * cfg.B * cfg.Hq
        tf = cfg.flops() / (ms / 1e3) / 1e12
        tf_exact = exact / (ms / 1e3) / 1e12
        out[cfg.name] = {
            "shape": {"B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "N": cfg.N_q, "d": cfg.d,
                      "dtype": cfg.dtype, "causal": cfg.causal,
                      "q_scale": 2 ** cfg.q_scale_pow2},
            "launches": n_launch if flushed else 3 * n_launch,
            "l2": ("256 MB written before each launch (inputs fit in L2)" if flushed else
                   f"back-to-back launches: inputs ({in_bytes / 1e6:.0f} MB) larger than L2"),
            "ms_per_launch": round(ms, 5),
            "ms_min": round(times[0], 5),
            "ms_median": round(times[len(times) // 2], 5),
            "flops_per_launch": cfg.flops(),
            "flops_exact_per_launch": exact,
            "value": round(tf, 1),
            "value_exact": round(tf_exact, 1),
            "unit": "TFLOP/s",
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                         "peak_source": f"{peak_src} bf16 burst (cuBLAS); fp16 nominal rate = bf16",
                         "frac": round(tf / peaks["bf16_tflops"], 4),
                         "frac_exact": round(tf_exact / peaks["bf16_tflops"], 4),
                         "frac_of_spec_2250": round(tf / 2250.0, 4)},
        }
        if cfg.N_q <= 256:
            out[cfg.name]["note"] = ("two 128-row query tiles on 152 SMs: launch- and latency-"
                                     "bound; the time is the figure, the fraction is not meaningful")
        del q, k, v, o, lse
    del flush
    return out


def measure_variants(args, attn, pcfg, q, k, v, o, lse, stream, peaks, peak_src):
    """The prefill variants that change the operator, on the same inputs: the pages' sliding
    window (W = 1024) and a block pattern.  TFLOP/s from the exact visible (query, key) pairs
    (4*d FLOPs each); timed with CUDA events over args.steps launches after 3 warm-ups."""
    import torch

    W = 1024
    import synthetic as syn

    pattern = syn.causal_block_pattern(pcfg.N_q, pcfg.N_kv)
    mask = torch.from_numpy(pattern).to(q.device)
    per_head = {
        "window": visible_keys_window(pcfg.N_q, pcfg.N_kv, W).sum(),
        "block_sparse": visible_keys_blocks(pcfg.N_q, pcfg.N_kv, pattern, True).sum(),
    }
    calls = {
        "window": lambda: attn.attn_fwd_window(q, k, v, W, o=o, lse=lse, scale=pcfg.scale,
                                                stream=stream),
        "block_sparse": lambda: attn.attn_fwd_block_sparse(q, k, v, mask, causal=True, o=o, lse=lse,
                                                           scale=pcfg.scale, stream=stream),
    }
    # backward of the same prefill: dO drawn on the device, the forward's own O and L
    dout = torch.randn(q.shape, device=q.device, generator=torch.Generator(q.device).manual_seed(77),
                       dtype=torch.float32).to(q.dtype)
    attn.attn_fwd(q, k, v, o=o, lse=lse, causal=True, scale=pcfg.scale, stream=stream)
    dq_b, dk_b, dv_b = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws_b = torch.empty(max(1, attn.attn_bwd_workspace_bytes(pcfg.B, pcfg.Hq, pcfg.N_q)),
                       device=q.device, dtype=torch.uint8)
    o_fwd, lse_fwd = o.clone(), lse.clone()
    calls["backward"] = lambda: attn.attn_bwd(q, k, v, o_fwd, dout, lse_fwd, causal=True,
                                              scale=pcfg.scale, dq=dq_b, dk=dk_b, dv=dv_b,
                                              workspace=ws_b, stream=stream)
    # FP8 with incoherent processing: rotation, block quantisation and attention per launch
    import synthetic as syn

    signs = torch.from_numpy(syn.random_signs(pcfg.d, 79)).to(q.device)
    ws_f8 = torch.empty(attn.attn_fwd_fp8_workspace_bytes(pcfg.B, pcfg.Hq, pcfg.Hkv, pcfg.N_q,
                                                          pcfg.N_kv, pcfg.d),
                        device=q.device, dtype=torch.uint8)
    calls["fp8"] = lambda: attn.attn_fwd_fp8(q, k, v, signs, o=o, lse=lse, causal=True,
                                             scale=pcfg.scale, workspace=ws_f8, stream=stream)
    out = {}
    for name, fn in calls.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        st = attn.attn_poll_status()
        if st != 0:
            raise SystemExit(f"device status after {name}: {attn.attn_status_string(st)}")
        ms = e0.elapsed_time(e1) / args.steps
        peak, peak_note = peaks["bf16_tflops"], f"{peak_src} bf16 burst (cuBLAS)"
        if name == "backward":
            # the pages' count: five matmuls against the forward's two (2.5x its FLOPs)
            flops = 2.5 * pcfg.flops()
        elif name == "fp8":
            flops = pcfg.flops()
            # E4M3 tensor rate: the bf16 measurement times the nominal ratio 4.5 / 2.25
            peak, peak_note = 2.0 * peak, f"{peak_src} bf16 burst (cuBLAS) x 2 (nominal fp8/bf16)"
        else:
            flops = 4.0 * pcfg.d * float(per_head[name]) * pcfg.B * pcfg.Hq
        tf = flops / (ms / 1e3) / 1e12
        out[name] = {
            "workload": (f"sliding window W={W}" if name == "window" else
                         f"causal block pattern, {int(pattern.sum())} of {pattern.size} blocks"
                         if name == "block_sparse" else
                         "backward (dQ, dK, dV) of the causal GQA prefill, FLOPs by the pages' "
                         "5-matmul count (2.5x forward)" if name == "backward" else
                         "causal prefill in FP8 (E4M3) with a randomised Hadamard rotation of Q "
                         "and K; each launch includes the rotation and quantisation")
                        + f" on the prefill workload's inputs; {args.steps} launches timed",
            "ms_per_launch": round(ms, 4), "flops_per_launch": flops, "value": round(tf, 1),
            "unit": "TFLOP/s",
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak,
                         "peak_source": peak_note, "frac": round(tf / peak, 4)},
        }
    return out


def measure_paged(args, attn, syn, dcfg, dq, dk, dv, do, dl, ws, lengths, max_len, dec_bytes,
                  stream, peaks, peak_src):
    """The decode step over a paged cache: the same cache scattered into shuffled 16-token
    pages (vLLM's default block size) and read through the block table.  GB/s of the same
    algorithmic bytes as the packed decode; timed like the variants."""
    import torch

    out = {}
    for page_size in (16, 128):
        table, n_pages, pg, sl = syn.paged_layout(lengths, page_size, seed=page_size)
        kp = syn.scatter_to_pages(dk, n_pages, page_size, pg, sl)
        vp = syn.scatter_to_pages(dv, n_pages, page_size, pg, sl)
        tbl = torch.from_numpy(table).to(dq.device)
        seq = torch.from_numpy(lengths.astype(np.int32)).to(dq.device)
        fn = lambda: attn.attn_decode_paged(dq, kp, vp, tbl, seq, max_len, o=do, lse=dl,
                                            split_size=dcfg.split, scale=dcfg.scale, workspace=ws,
                                            stream=stream)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        st = attn.attn_poll_status()
        if st != 0:
            raise SystemExit(f"device status after paged decode: {attn.attn_status_string(st)}")
        ms = e0.elapsed_time(e1) / args.steps
        gbs = dec_bytes / (ms / 1e3) / 1e9
        out[f"page_{page_size}"] = {
            "workload": f"the decode workload in shuffled {page_size}-token pages ({n_pages} pages)",
            "ms_per_launch": round(ms, 4), "value": round(gbs, 1), "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                         "peak_source": f"{peak_src} HBM copy",
                         "frac": round(gbs / peaks["hbm_gbs"], 4)},
        }
        del kp, vp
    return out


def run_e2e(args, attn, pcfg, q, k, v, stream, device, world):
    """The prefill from pinned host buffers to pinned host buffers: every step copies Q, K, V
    in, runs attn_fwd and copies O and L out.  Two steps are in flight, as in a serving loop:
    the inputs of step i + 1 go up (one stream) while step i computes (another) and step i - 1's
    result comes down (a third), on two sets of device buffers."""
    import torch

    hq = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    hk = torch.empty(k.shape, dtype=k.dtype, pin_memory=True)
    hv = torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
    hq.copy_(q)
    hk.copy_(k)
    hv.copy_(v)
    ho = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    hl = torch.empty((pcfg.B, pcfg.Hq, pcfg.N_q), dtype=torch.float32, pin_memory=True)
    sets = [(torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(q),
             torch.empty((pcfg.B, pcfg.Hq, pcfg.N_q), device=device, dtype=torch.float32))
            for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    s_cmp = stream
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]
    steps = max(3, min(args.steps, 20))

    def step(i):
        b = i % 2
        dq, dk, dv, do, dl = sets[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_cmp[b])  # step i - 2 has finished reading these inputs
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            ev_in[b].record(s_in)
        s_cmp.wait_event(ev_in[b])
        if used[b]:
            s_cmp.wait_event(ev_out[b])  # step i - 2's result has left these buffers
        attn.attn_fwd(dq, dk, dv, o=do, lse=dl, causal=True, scale=pcfg.scale, stream=s_cmp)
        ev_cmp[b].record(s_cmp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[b])
            ho.copy_(do, non_blocking=True)
            hl.copy_(dl, non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    barrier(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)  # every timed copy and launch is ordered after this
    for i in range(steps):
        step(3 + i)
    e1.record(s_out)  # the last step's result is on the host when this completes
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)

    # the same steps one at a time on one stream: copies in, the call, copies out
    dq, dk, dv, do, dl = sets[0]

    def serial_step():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        attn.attn_fwd(dq, dk, dv, o=do, lse=dl, causal=True, scale=pcfg.scale, stream=s_cmp)
        ho.copy_(do, non_blocking=True)
        hl.copy_(dl, non_blocking=True)

    with torch.cuda.stream(s_cmp):
        serial_step()
        torch.cuda.synchronize()
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(s_cmp)
        for _ in range(steps):
            serial_step()
        e3.record(s_cmp)
    torch.cuda.synchronize()
    ms_serial = e2.elapsed_time(e3)
    ms_max, ms_serial_max = reduce_max([ms, ms_serial], device)
    h2d = (q.numel() + k.numel() + v.numel()) * 2
    d2h = q.numel() * 2 + pcfg.B * pcfg.Hq * pcfg.N_q * 4
    return {
        "value": round(pcfg.flops() * steps * world / (ms_max / 1e3) / 1e12, 2),
        "unit": "TFLOP/s",
        "h2d_bytes_per_step": int(h2d),
        "d2h_bytes_per_step": int(d2h),
        "steps": steps,
        "ms_per_step": round(ms_max / steps, 4),
        "pipeline": "two steps in flight: inputs up, compute and result down on three streams",
        "serial": {
            "value": round(pcfg.flops() * steps * world / (ms_serial_max / 1e3) / 1e12, 2),
            "unit": "TFLOP/s",
            "ms_per_step": round(ms_serial_max / steps, 4),
            "pipeline": "one step at a time on one stream (copies in, call, copies out)",
        },
    }


def run_e2e_decode(args, attn, dcfg, dq, dk, dv, cu, max_len, ws, dec_bytes, stream, device,
                   world):
    """The decode step from pinned host buffers: every step copies the new query token of every
    sequence and the sequence offsets up, runs attn_decode_splitkv over the resident KV cache
    (the cache is the server's state, not a per-step input) and copies O and L down; one step
    at a time on one stream.  GB/s of the same algorithmic bytes as the device-resident line."""
    import torch

    hq = torch.empty(dq.shape, dtype=dq.dtype, pin_memory=True)
    hq.copy_(dq)
    hcu = torch.empty(cu.shape, dtype=cu.dtype, pin_memory=True)
    hcu.copy_(cu)
    ho = torch.empty(dq.shape, dtype=dq.dtype, pin_memory=True)
    hl = torch.empty((dcfg.B, dcfg.Hq), dtype=torch.float32, pin_memory=True)
    q_d, cu_d, o_d = torch.empty_like(dq), torch.empty_like(cu), torch.empty_like(dq)
    l_d = torch.empty((dcfg.B, dcfg.Hq), device=device, dtype=torch.float32)
    steps = max(3, min(args.steps, 50))

    def step():
        q_d.copy_(hq, non_blocking=True)
        cu_d.copy_(hcu, non_blocking=True)
        attn.attn_decode_splitkv(q_d, dk, dv, cu_d, max_len, o=o_d, lse=l_d,
                                 split_size=dcfg.split, scale=dcfg.scale, workspace=ws,
                                 stream=stream)
        ho.copy_(o_d, non_blocking=True)
        hl.copy_(l_d, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        barrier(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
    torch.cuda.synchronize()
    (ms_max,) = reduce_max([e0.elapsed_time(e1)], device)
    return {
        "value": round(dec_bytes * steps * world / (ms_max / 1e3) / 1e9, 1),
        "unit": "GB/s",
        "h2d_bytes_per_step": int(hq.numel() * 2 + hcu.numel() * 4),
        "d2h_bytes_per_step": int(ho.numel() * 2 + hl.numel() * 4),
        "steps": steps,
        "ms_per_step": round(ms_max / steps, 4),
        "pipeline": "one step at a time on one stream; the KV cache stays resident",
    }


def cpu_baseline_prefill(pcfg, q, k, v, budget_s=12.0):
    import oracle
    import synthetic as syn

    qb, kb, vb = (syn.tensor_to_bits(t) for t in (q, k, v))
    tflops, n_rows, t = time_oracle_prefill(pcfg, qb, kb, vb, budget_s)
    return {
        "value": round(tflops, 6),
        "unit": "TFLOP/s",
        "cores": oracle.max_threads(),
        "kind": "oracle",
        "sample": f"{n_rows} random query rows of the prefill workload in calls of 1024 rows "
                  f"({t:.1f} s, exact per-row FLOPs 4*d*visible keys), fp64",
    }


# ----------------------------------------------------------------------------------------
# reference arm: the oracle as it stands, on the host cores
# ----------------------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import synthetic as syn

    pcfg = syn.CONFIG4
    q, k, v = pcfg.host_inputs()
    # 1024 rows a step: the oracle's fixed cost per call (about 75 ms) stays a small part of
    # the step, so the line reports the oracle's throughput rather than its call overhead
    rows_per_step = 1024
    for i in range(args.warmup):
        oracle.attention_rows(q, k, v, pcfg.dtype, pcfg.B, pcfg.Hq, pcfg.Hkv, pcfg.N_q, pcfg.N_kv,
                              pcfg.d, True, pcfg.scale, prefill_sample_rows(pcfg, rows_per_step, 10_000 + i))
    flops, t = 0.0, 0.0
    for i in range(args.steps):
        rows = prefill_sample_rows(pcfg, rows_per_step, i)
        t0 = time.perf_counter()
        oracle.attention_rows(q, k, v, pcfg.dtype, pcfg.B, pcfg.Hq, pcfg.Hkv, pcfg.N_q, pcfg.N_kv,
                              pcfg.d, True, pcfg.scale, rows)
        t += time.perf_counter() - t0
        flops += row_flops(pcfg, rows)
    value = flops / t / 1e12
    sample = (f"{rows_per_step} random query rows of the prefill workload per step "
              f"(exact per-row FLOPs), fp64 oracle")
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1), drawn on host)",
        "config": {"workload": "gqa causal prefill B=1 Hq=64 Hkv=8 N=8192 d=128 bf16 (sampled rows)",
                   "prefill": pcfg.name},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the sliding-window and block-sparse prefill measurements")
    ap.add_argument("--only", choices=["both", "prefill", "decode", "configs"], default="both",
                    help="run one half of the step, or only the table of other prefill "
                         "workloads (for profiling)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the table of other prefill workloads")
    ap.add_argument("--config", default=None,
                    help="time only this workload of the table (a name from synthetic.py)")
    ap.add_argument("--decode-batch", type=int, default=64,
                    help="sequences of the decode workload (first B of the seeded lengths)")
    ap.add_argument("--prefill-heads", type=int, default=64,
                    help="query heads of the prefill workload (the key/value heads follow the "
                         "group size; fewer heads make a smaller case for profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

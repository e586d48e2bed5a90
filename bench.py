"""Benchmark: exact-attention forward TFLOP/s and flash-decoding GB/s on GB300.

One step = one pass of the whole hot path over one batch of synthetic input,
on the largest single-GPU configurations of the workloads below:
  prefill  attn_fwd   long_sequence: B=1, Hq=32, Hkv=8, Nq=Nk=16384, d=128,
                      causal, bf16 (the sequence-parallel stress shape)
  decode   attn_decode_splitkv  decode_b16_8k: B=16, Hq=32, Hkv=8, Nk=8192,
                      d=128, bf16 (split-KV with the automatic segment count)
Every other workload (single head fp32/bf16, ragged d=64 causal and
non-causal, the q x 8 outlier variants, training-style prefill, the 64K-key
decode) is timed the same way and reported per workload under "configs".
Inputs are resident in HBM when a timed call starts; L2 is flushed before
every timed call, outside the events: a 256 MiB write and then a 512 MiB
read, so that L2 holds only clean lines of another buffer and no write-back
of the flush (or of the previous call's output) lands inside the timed
region.  (A read of 256 MiB, twice the L2, still left dirty lines whose
write-back measured 2 us on the 64K-key decode and 4 us on B16 x 8K.)  Each call is timed with CUDA events on the launching stream.

value  = prefill TFLOP/s (FLOPs counted as 4 Nq Nk d per head, halved for
         causal, summed over ranks) / max-over-ranks time.
decode = GB/s of the decode call (K + V + Q + O + LSE bytes, each once).
e2e    = the same metrics through the C ABI with pinned host buffers: the
         host->device copy of the inputs and the device->host copy of O and
         LSE are inside the timed region (the forward through attn_fwd_host,
         the decode through attn_decode_splitkv after its copies).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 run under torchrun; every rank runs an independent replica of the
workload (weak scaling) and rank 0 prints the line.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s & % of GB300 BF16 tensor peak; decode GB/s & % of HBM BW"

# name -> (B, Hq, Hkv, Nq, Nk, d, causal)
PREFILL = {
    "single_head": (1, 1, 1, 256, 256, 64, False),
    "ragged": (8, 12, 12, 1000, 1000, 64, False),
    "ragged_causal": (8, 12, 12, 1000, 1000, 64, True),
    "training_prefill": (4, 16, 16, 4096, 4096, 128, True),
    "long_sequence": (1, 32, 8, 16384, 16384, 128, True),
    # d = 64 versions of the two large shapes (for measuring the d = 64 kernel;
    # not workloads of the report)
    "training_prefill_d64": (4, 16, 16, 4096, 4096, 64, True),
    "long_sequence_d64": (1, 32, 8, 16384, 16384, 64, True),
}
DECODE = {
    "decode_64k": (1, 32, 8, 65536, 128),
    "decode_b16_8k": (16, 32, 8, 8192, 128),
}

# The step's workloads (the largest single-GPU configurations).
HEADLINE_PREFILL = "long_sequence"
HEADLINE_DECODE = "decode_b16_8k"

# Every workload reported under "configs": name -> (prefill shape, dtype, q scale).
PREFILL_CONFIGS = {
    "single_head_fp32": ("single_head", "float32", 1.0),
    "single_head_bf16": ("single_head", "bfloat16", 1.0),
    "ragged": ("ragged", "bfloat16", 1.0),
    "ragged_causal": ("ragged_causal", "bfloat16", 1.0),
    "ragged_outlier": ("ragged", "bfloat16", 8.0),
    "ragged_outlier_causal": ("ragged_causal", "bfloat16", 8.0),
    "training_prefill": ("training_prefill", "bfloat16", 1.0),
    "long_sequence": ("long_sequence", "bfloat16", 1.0),
}
NOMINAL_HBM_GBS = 8000.0  # the ~8 TB/s HBM3e figure the decode target is quoted against

# DRAM traffic of one launch from an ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by the hash of the kernel source it was
# measured on: any later change to the source turns the figure into null.
NCU_TRAFFIC = {
    "long_sequence": {"bytes_per_launch": 350.80e6 + 101.38e6, "src": "fwd_tc.cu",
                      "src_hash": "f289683a689bd204"},
    "decode_b16_8k": {"bytes_per_launch": 537.03e6 + 2.67e6, "src": "decode.cu",
                      "src_hash": "38855097fe3c6171"},
}

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def prefill_flops(cfg) -> float:
    B, Hq, Hkv, Nq, Nk, d, causal = cfg
    f = 4.0 * Nq * Nk * d * B * Hq
    return f / 2 if causal else f


def decode_bytes(cfg) -> float:
    B, Hq, Hkv, Nk, d = cfg
    kv = 2.0 * B * Nk * Hkv * d * 2
    return kv + 2.0 * B * Hq * d * 2 + B * Hq * 4


def src_hash(name: str) -> str:
    p = os.path.join(ROOT, "exact_attention_62_gb300", "csrc", name)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples nvidia-smi clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return
        t0 = time.time()  # wait for the first sample so the window is covered
        while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def whole_job_rate(work_per_rank: float, ms_max_over_ranks: float, world: int, scale: float) -> float:
    """Weak scaling: every rank runs the same workload as an independent
    replica, so the job's throughput is all ranks' work over the slowest
    rank's time (`scale` converts units/s to the reported unit)."""
    return work_per_rank * world / (ms_max_over_ranks * 1e-3) / scale


def prefill_desc(name: str) -> str:
    B, Hq, Hkv, Nq, Nk, d, causal = PREFILL[name]
    return "%s (B=%d Hq=%d Hkv=%d Nq=%d Nk=%d d=%d %s)" % (
        name, B, Hq, Hkv, Nq, Nk, d, "causal" if causal else "non-causal")


def decode_desc(name: str) -> str:
    B, Hq, Hkv, Nk, d = DECODE[name]
    return "%s (B=%d Hq=%d Hkv=%d Nk=%d d=%d)" % (name, B, Hq, Hkv, Nk, d)


def workload_config(args) -> dict:
    """The step's workload, the same on both arms."""
    return {
        "workload": "prefill %s + decode %s, bf16" % (prefill_desc(args.prefill), decode_desc(args.decode)),
        "l2": "inputs larger than L2; L2 flushed before every timed call (256 MiB write, then "
              "512 MiB read so no dirty line is written back inside the timed region)",
    }


# ----------------------------------------------------------------------------- reference arm

_ORACLE_INPUTS = {}


def oracle_prefill_sample(cfg, seconds: float, seed: int = 0):
    """Times the oracle (as it stands) on random rows of the prefill workload
    until `seconds` of wall time are used.  Returns (TFLOP/s, rows, cores)."""
    import oracle
    from exact_attention_62_gb300.inputs import make_qkv, sample_rows
    B, Hq, Hkv, Nq, Nk, d, causal = cfg
    key = (cfg, seed)
    if key not in _ORACLE_INPUTS:
        q, k, v = make_qkv(B, Hq, Hkv, Nq, Nk, d, seed)
        _ORACLE_INPUTS[key] = (tuple(oracle._f32(x) for x in (q, k, v)),
                               sample_rows(B, Hq, Nq, 1 << 20, seed + 1))
    (qf, kf, vf), rows = _ORACLE_INPUTS[key]
    per_row = prefill_flops(cfg) / (B * Hq * Nq)  # same counting as the GPU metric
    done, t_used, chunk = 0, 0.0, 256
    while t_used < seconds and done < len(rows):
        sel = rows[done:done + chunk]
        t0 = time.perf_counter()
        oracle.attn_rows(qf, kf, vf, causal, 1.0 / math.sqrt(d), sel)
        t_used += time.perf_counter() - t0
        done += len(sel)
        chunk = min(chunk * 2, 8192)
    return done * per_row / t_used / 1e12, done, oracle.num_threads()


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    cfg = PREFILL[args.prefill]
    per_step = max(1.0, min(8.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_prefill_sample(cfg, per_step / 4)
    vals, rows_total, cores = [], 0, 1
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, rows, cores = oracle_prefill_sample(cfg, per_step)
        vals.append(v)
        rows_total += rows
    wall = time.perf_counter() - t0
    value = statistics.mean(vals)
    B, Hq, Hkv, Nq, Nk, d, causal = cfg
    sample = ("%d random rows (b, hq, i) of the %s prefill per step, ~%.0f s of CPU work each; "
              "FLOPs counted as for the GPU (4 Nk d per row, halved for causal); the oracle is "
              "timed on the prefill half of the step, whose FLOPs are the metric") % (
        rows_total // max(1, args.steps), args.prefill, per_step)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * wall / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- our arm

def _timed_ms(call, reps: int, flush, warmup: int = 3) -> float:
    """Mean CUDA-event time of `call` over `reps` calls, L2 flushed before each."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush()
        call()
    ts = []
    for _ in range(reps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        ts.append((e0, e1))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ts)


def measure_configs(attn, dev, flush, reps: int, peaks) -> dict:
    """Every workload timed alone (L2 flushed before each call), with its
    throughput and roofline fraction."""
    import torch
    from exact_attention_62_gb300.inputs import make_qkv
    peak_t, peak_h = float(peaks["bf16_tflops"]), float(peaks["hbm_gbs"])
    out = {}
    for name, (shape, dt, q_scale) in PREFILL_CONFIGS.items():
        B, Hq, Hkv, Nq, Nk, d, causal = PREFILL[shape]
        dtype = getattr(torch, dt)
        q, k, v = (x.to(dev) for x in make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=30, dtype=dtype,
                                                 q_scale=q_scale))
        o, lse = torch.empty_like(q), torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
        scale = 1.0 / math.sqrt(d)
        ms = _timed_ms(lambda: attn.attn_fwd(q, k, v, causal, scale, o=o, lse=lse), reps, flush)
        tf = prefill_flops(PREFILL[shape]) / (ms * 1e-3) / 1e12
        entry = {"shape": prefill_desc(shape), "dtype": dt, "ms": ms, "value": tf, "unit": "TFLOP/s"}
        if q_scale != 1.0:
            entry["q_scale"] = q_scale
        if shape == "single_head":
            entry["frac"] = None
            entry["note"] = "latency-bound (one 256-row unit on one SM): time only"
        elif dt == "bfloat16":
            entry["frac"] = tf / peak_t
            entry["peak"] = peak_t
        out[name] = entry
        del q, k, v, o, lse
    for name in ("decode_64k", "decode_b16_8k"):
        B, Hq, Hkv, Nk, d = DECODE[name]
        q, k, v = (x.to(dev) for x in make_qkv(B, Hq, Hkv, 1, Nk, d, seed=31))
        S = attn.attn_decode_num_splits(B, Hq, Hkv, Nk, d)
        ws = torch.empty(max(16, attn.attn_decode_workspace_bytes(B, Hq, Hkv, Nk, d, S)),
                         dtype=torch.uint8, device=dev)
        o, lse = torch.empty_like(q), torch.empty((B, Hq), dtype=torch.float32, device=dev)
        scale = 1.0 / math.sqrt(d)
        ms = _timed_ms(lambda: attn.attn_decode_splitkv(q, k, v, scale, S, workspace=ws, o=o, lse=lse),
                       reps, flush)
        gbs = decode_bytes(DECODE[name]) / (ms * 1e-3) / 1e9
        out[name] = {"shape": decode_desc(name), "dtype": "bfloat16", "splits": S, "ms": ms,
                     "value": gbs, "unit": "GB/s", "frac": gbs / peak_h, "peak": peak_h,
                     "frac_of_nominal_8tbs": gbs / NOMINAL_HBM_GBS}
        del q, k, v, o, lse, ws
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_attention_62_gb300 as attn
    from exact_attention_62_gb300.inputs import make_qkv

    attn.ensure_built()
    do_pre = args.only in (None, "prefill")
    do_dec = args.only in (None, "decode")
    pcfg = PREFILL[args.prefill]
    dcfg = DECODE[args.decode]
    B, Hq, Hkv, Nq, Nk, d, causal = pcfg
    dB, dHq, dHkv, dNk, dd = dcfg
    stream = torch.cuda.current_stream()
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(128 << 20, dtype=torch.float32, device=dev)

    def flush_l2():
        # The write evicts everything; the read, four times the L2, then
        # replaces the dirty lines with clean ones, so their write-back happens
        # here and not later.
        flush_w.zero_()
        flush_r.sum()

    if do_pre:
        scale = 1.0 / math.sqrt(d)
        qh, kh, vh = make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=10 + rank)
        q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    if do_dec:
        dq_h, dk_h, dv_h = make_qkv(dB, dHq, dHkv, 1, dNk, dd, seed=20 + rank)
        dq, dk, dv = dq_h.to(dev), dk_h.to(dev), dv_h.to(dev)
        splits = attn.attn_decode_num_splits(dB, dHq, dHkv, dNk, dd)
        if args.splits:
            splits = args.splits
        wbytes = attn.attn_decode_workspace_bytes(dB, dHq, dHkv, dNk, dd, splits)
        ws = torch.empty(max(16, wbytes), dtype=torch.uint8, device=dev)
        do = torch.empty_like(dq)
        dlse = torch.empty((dB, dHq), dtype=torch.float32, device=dev)

    def prefill():
        if do_pre:
            attn.attn_fwd(q, k, v, causal, scale, o=o, lse=lse)

    def decode():
        if do_dec:
            attn.attn_decode_splitkv(dq, dk, dv, 1.0 / math.sqrt(dd), splits, workspace=ws,
                                     o=do, lse=dlse)

    for _ in range(args.warmup):
        flush_l2()
        prefill()
        decode()
    torch.cuda.synchronize()
    if attn.attn_check_device_status() != 0:
        raise RuntimeError("device status reports a timed-out wait during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    # The timed region lasts milliseconds, shorter than nvidia-smi's sampling
    # period, so the same step also runs untimed for ~0.5 s right before it:
    # the clock samples cover that soak and the timed region.
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < 0.5:
        for _ in range(8):
            prefill()
            decode()
        torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for s in range(K):
        flush_l2()
        ev[s][0].record(stream)
        prefill()
        ev[s][1].record(stream)
        flush_l2()
        ev[s][2].record(stream)
        decode()
        ev[s][3].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    if attn.attn_check_device_status() != 0:
        raise RuntimeError("device status reports a timed-out wait")
    pre_total = max_over_ranks(sum(ev[s][0].elapsed_time(ev[s][1]) for s in range(K)), world, dev)
    dec_total = max_over_ranks(sum(ev[s][2].elapsed_time(ev[s][3]) for s in range(K)), world, dev)
    peaks, peak_src = load_peaks()

    if args.only is not None:
        if rank == 0:
            print(json.dumps({"profile_only": args.only, "prefill_ms": pre_total / K,
                              "decode_ms": dec_total / K, "clocks": clk}))
        return 0

    # ---- every workload of the method, each timed alone (rank 0's GPU)
    configs = None
    if not args.no_configs and rank == 0:
        configs = measure_configs(attn, dev, flush_l2, min(K, 20), peaks)
        if attn.attn_check_device_status() != 0:
            raise RuntimeError("device status reports a timed-out wait")

    # ---- end to end through the C ABI with pinned host buffers
    e_pre_ms = e_dec_ms = None
    if not args.no_e2e:
        qh_p, kh_p, vh_p = qh.pin_memory(), kh.pin_memory(), vh.pin_memory()
        o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        l_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        dq_p, dk_p, dv_p = dq_h.pin_memory(), dk_h.pin_memory(), dv_h.pin_memory()
        do_h = torch.empty(do.shape, dtype=do.dtype).pin_memory()
        dl_h = torch.empty(dlse.shape, dtype=dlse.dtype).pin_memory()
        e_pre, e_dec = [], []
        # the forward through attn_fwd_host: chunks copied in, computed and
        # copied back on three streams, the transfers overlapping the computation
        # (the default chunking: sixteen row chunks for one sequence)
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        for s in range(max(3, min(K, 10)) + 1):
            flush_l2()
            e0, e1, e2, e3 = (torch.cuda.Event(enable_timing=True) for _ in range(4))
            e0.record(stream)
            if do_pre:
                attn.attn_fwd_host(qh_p, kh_p, vh_p, causal, scale, o=o_h, lse=l_h,
                                   device_buffers=(q, k, v, o, lse), stream=stream,
                                   h2d_stream=up, d2h_stream=down)
            e1.record(stream)
            flush_l2()
            e2.record(stream)
            dq.copy_(dq_p, non_blocking=True)
            dk.copy_(dk_p, non_blocking=True)
            dv.copy_(dv_p, non_blocking=True)
            decode()
            do_h.copy_(do, non_blocking=True)
            dl_h.copy_(dlse, non_blocking=True)
            e3.record(stream)
            torch.cuda.synchronize()
            if s > 0:  # the first pass warms the copy path
                e_pre.append(e0.elapsed_time(e1))
                e_dec.append(e2.elapsed_time(e3))
        e_pre_ms = max_over_ranks(statistics.mean(e_pre), world, dev)
        e_dec_ms = max_over_ranks(statistics.mean(e_dec), world, dev)

    # ---- roofline of the forward kernel (the step's dominant kernel) and of decode
    flops = prefill_flops(pcfg)
    pre_ms_avg = pre_total / K
    achieved = flops / (pre_ms_avg * 1e-3) / 1e12
    peak_t = float(peaks["bf16_tflops"])

    def traffic_of(name):
        rec = NCU_TRAFFIC.get(name)
        if not rec or rec.get("bytes_per_launch") is None:
            return None
        return rec["bytes_per_launch"] if rec.get("src_hash") == src_hash(rec["src"]) else None

    traffic = traffic_of(args.prefill)
    dbytes = decode_bytes(dcfg)
    dec_ms_avg = dec_total / K
    dec_gbs = dbytes / (dec_ms_avg * 1e-3) / 1e9
    peak_h = float(peaks["hbm_gbs"])
    dtraffic = traffic_of(args.decode)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0
    cpu = None
    if not args.no_cpu_baseline:
        v_cpu, rows, cores = oracle_prefill_sample(pcfg, args.cpu_seconds)
        cpu = {"value": v_cpu, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": "%d random rows of the %s prefill (~%.0f s of CPU work), FLOPs counted "
                         "as for the GPU (4 Nk d per row, halved for causal)"
                         % (rows, args.prefill, args.cpu_seconds)}
    launches_per_step = 1 + (1 if splits == 1 else 2)
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
    dh2d = sum(t.numel() * t.element_size() for t in (dq, dk, dv))
    dd2h = do.numel() * do.element_size() + dlse.numel() * dlse.element_size()
    e2e = None
    de2e = None
    if e_pre_ms is not None:
        e2e = {"value": whole_job_rate(flops, e_pre_ms, world, 1e12), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": "attn_fwd_host: host copies overlapping the forward"}
        de2e = {"value": whole_job_rate(dbytes, e_dec_ms, world, 1e9), "unit": "GB/s",
                "h2d_bytes_per_step": dh2d, "d2h_bytes_per_step": dd2h}
    config = workload_config(args)
    config.update({
        "prefill": {"B": B, "Hq": Hq, "Hkv": Hkv, "Nq": Nq, "Nk": Nk, "d": d,
                    "causal": bool(causal), "ms": pre_ms_avg},
        "decode": {"B": dB, "Hq": dHq, "Hkv": dHkv, "Nk": dNk, "d": dd, "splits": splits,
                   "ms": dec_ms_avg},
        "parallelism": "independent replicas" if world > 1 else "single GPU",
        "clocks_window": "nvidia-smi every 100 ms over a 0.5 s untimed soak of the same "
                         "step followed by the timed steps",
    })
    line = {
        "metric": METRIC,
        "value": whole_job_rate(flops, pre_ms_avg, world, 1e12),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": (pre_total + dec_total) / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": config,
        "decode": {
            "value": whole_job_rate(dbytes, dec_ms_avg, world, 1e9), "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": peak_h, "unit": "GB/s",
                         "frac": dec_gbs / peak_h, "traffic": dtraffic,
                         "peak_source": "%s HBM copy" % peak_src,
                         "frac_of_nominal_8tbs": dec_gbs / NOMINAL_HBM_GBS},
            "e2e": de2e,
        },
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                     "frac": achieved / peak_t, "traffic": traffic,
                     "peak_source": "%s bf16 burst" % peak_src},
        "e2e": e2e,
        "cpu_baseline": cpu,
        "clocks": clk,
        "gpu_launches": K * launches_per_step,
        "configs": configs,
        "wall_s": t_wall,
    }
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_extra(args):
    """--only backward / fp8: attn_bwd or attn_fwd_fp8 on the prefill workload;
    --only paged: attn_decode_paged on the decode workload with pages of
    --page-size keys in a random order.  Timed like the step's calls (L2
    flushed clean before each, CUDA events).  For profiling; prints one JSON
    line, not the bench contract."""
    import torch
    import exact_attention_62_gb300 as attn
    from exact_attention_62_gb300.inputs import make_paged, make_qkv
    attn.ensure_built()
    dev = torch.device("cuda", 0)
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush_r = torch.ones(128 << 20, dtype=torch.float32, device=dev)
    if args.only == "paged":
        dB, dHq, dHkv, dNk, dd = DECODE[args.decode]
        qh, kp, vp, table, lens = make_paged(dB, dHq, dHkv, dd, args.page_size, [dNk] * dB, seed=20,
                                             extra_pages=0, poison=False)
        qh, kp, vp, table, lens = (x.to(dev) for x in (qh, kp, vp, table, lens))
        call = lambda: attn.attn_decode_paged(qh, kp, vp, table, lens, dNk, 1.0 / math.sqrt(dd))
        return _time_extra(args, call, flush_w, flush_r, attn, "GB/s", decode_bytes(DECODE[args.decode]) / 1e9,
                           args.decode)
    if args.only == "splitkv":
        dB, dHq, dHkv, dNk, dd = DECODE[args.decode]
        qh, kh, vh = (x.to(dev) for x in make_qkv(dB, dHq, dHkv, 1, dNk, dd, seed=20))
        splits = args.splits or attn.attn_decode_num_splits(dB, dHq, dHkv, dNk, dd)
        ws = torch.empty(max(16, attn.attn_decode_workspace_bytes(dB, dHq, dHkv, dNk, dd, splits)),
                         dtype=torch.uint8, device=dev)
        do, dl = torch.empty_like(qh), torch.empty((dB, dHq), dtype=torch.float32, device=dev)
        call = lambda: attn.attn_decode_splitkv(qh, kh, vh, 1.0 / math.sqrt(dd), splits, workspace=ws,
                                                o=do, lse=dl)
        return _time_extra(args, call, flush_w, flush_r, attn, "GB/s", decode_bytes(DECODE[args.decode]) / 1e9,
                           args.decode, {"splits": splits})
    B, Hq, Hkv, Nq, Nk, d, causal = PREFILL[args.prefill]
    scale = 1.0 / math.sqrt(d)
    q, k, v = (x.to(dev) for x in make_qkv(B, Hq, Hkv, Nq, Nk, d, seed=10))
    o, lse = attn.attn_fwd(q, k, v, causal, scale)
    if args.only == "forward":
        call = lambda: attn.attn_fwd(q, k, v, causal, scale, o=o, lse=lse)
        return _time_extra(args, call, flush_w, flush_r, attn, "tflops",
                           prefill_flops(PREFILL[args.prefill]) / 1e12, args.prefill)
    if args.only == "backward":
        dout = torch.randn_like(q)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(attn.attn_bwd_workspace_bytes(B, Hq, Nq), dtype=torch.uint8, device=dev)
        call = lambda: attn.attn_bwd(q, k, v, o, lse, dout, causal, scale, dq=dq, dk=dk, dv=dv,
                                     workspace=ws)
        flops = 2.5 * prefill_flops(PREFILL[args.prefill])  # five products of 2 Nq Nk d per head
    elif args.only == "fp8pv":
        q8, qs = attn.attn_quantize_fp8(q)
        k8, ks = attn.attn_quantize_fp8(k)
        vt8, vs = attn.attn_quantize_fp8_v(v)
        call = lambda: attn.attn_fwd_fp8_pv(q8, k8, vt8, qs, ks, vs, causal, scale, o=o, lse=lse)
        flops = prefill_flops(PREFILL[args.prefill])
    else:
        q8, qs = attn.attn_quantize_fp8(q)
        k8, ks = attn.attn_quantize_fp8(k)
        call = lambda: attn.attn_fwd_fp8(q8, k8, v, qs, ks, causal, scale, o=o, lse=lse)
        flops = prefill_flops(PREFILL[args.prefill])
    return _time_extra(args, call, flush_w, flush_r, attn, "tflops", flops / 1e12, args.prefill)


def _time_extra(args, call, flush_w, flush_r, attn, unit, work, workload, extra=None):
    import torch
    for _ in range(args.warmup):
        flush_w.zero_()
        flush_r.sum()
        call()
    ts = []
    for _ in range(args.steps):
        flush_w.zero_()
        flush_r.sum()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    if attn.attn_check_device_status() != 0:
        raise RuntimeError("device status reports a timed-out wait")
    ms = statistics.mean(ts)
    out = {"profile_only": args.only, "workload": workload, "ms": ms, unit: work / (ms * 1e-3)}
    if args.only == "paged":
        out["page_size"] = args.page_size
    out.update(extra or {})
    print(json.dumps(out))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--prefill", choices=sorted(PREFILL), default=HEADLINE_PREFILL)
    ap.add_argument("--decode", choices=sorted(DECODE), default=HEADLINE_DECODE)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--page-size", type=int, default=16, help="--only paged: keys per page")
    ap.add_argument("--only", choices=["prefill", "decode", "forward", "splitkv", "backward", "fp8",
                                        "fp8pv", "paged"], default=None,
                    help="time one part only (for profiling; no JSON contract): a half of the "
                         "step with the clock soak (prefill, decode); or, without the soak, "
                         "attn_fwd / the backward pass / the FP8-Q,K forward / the FP8-Q,K,V "
                         "forward with e4m3 P on the prefill "
                         "workload, attn_decode_splitkv / the paged decode on the decode workload")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload block (every workload timed alone)")
    ap.add_argument("--splits", type=int, default=0, help="decode segments (0 = automatic)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.only in ("forward", "splitkv", "backward", "fp8", "fp8pv", "paged"):
        return run_extra(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the paged NVFP4 decode step on GB300.

One step = the whole decode path for one new token of the million-token
workload (1 sequence, 1,048,576 keys after the append, 24 query / 4 KV heads
of dim 256, YaRN x4, NVFP4 pool in 16-token pages randomly permuted):

    kv_append_nvfp4 -> paged_decode_attention -> split_kv_combine

(the YaRN table is built once, before timing).  ``value`` is KV tokens per
second per layer with inputs resident in HBM; the pool (1.2 GB) is far
larger than L2, so no flush is needed between steps.  ``e2e`` times the same
step through the public API with the step's inputs (q, k, v of the new
token) copied from pinned host memory and the bf16 output copied back.

``--impl reference`` times the CPU oracle (float64 NumPy) on the host cores
instead, on a bounded sample of the same workload.
"""
import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "1M-ctx paged decode attention: KV tokens/s/layer and HBM GB/s (% of GB300 peak)"
UNIT = "KV tokens/s/layer"
FALLBACK_HBM_GBS = 6800.0   # earlier GB300 copy measurement, used if no measured peaks file
ALGO_BYTES_PER_TOKEN = {"nvfp4": 4 * 2 * (128 + 16), "fp8": 4 * 2 * 256, "int8": 4 * 2 * (256 + 8),
                        "bf16": 4 * 2 * 256 * 2}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--config", type=int, default=3,
                   help="workload number: 1..5 as in the workload table, 6 = reduced chunked prefill "
                        "(profiling), 7/8 = the million-token decode with an FP8/INT8 cache, "
                        "9 = reduced multi-session verify (profiling)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--layers", type=int, default=16,
                   help="also time a CUDA-graph replay of this many layers' steps (per-token "
                        "latency); 1 skips it")
    p.add_argument("--fp4q", action="store_true",
                   help="prefill workloads: NVFP4-encoded queries (block-scaled FP4 QK^T, "
                        "paged_prefill_attention_fp4q) instead of bf16 queries")
    p.add_argument("--no-configs", action="store_true",
                   help="skip the other workloads' records (the 'configs' object)")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    return p.parse_args()


def replica_max(x, world, device):
    """Max of ``x`` over the ranks (the slowest replica sets the time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_rate(units_per_rank, ms, world):
    """Whole-job rate: the units all ranks processed over the max-over-ranks
    time (replicas each process the same workload)."""
    return world * units_per_rank / (ms * 1e-3)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBps", "hbm"):
            if key in d:
                return float(d[key]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


DECODE_SOURCES = ("decode.cu", "decode_common.cuh", "device_common.cuh")


def profiled_traffic(kv_dtype):
    """DRAM bytes per decode launch from the committed ncu summary, or None when
    the decode kernel's source changed since that capture."""
    import hashlib
    if kv_dtype != "nvfp4":
        return None
    path = os.path.join(ROOT, "profiles", "paged_decode_nvfp4_1M_keys.md")
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        line = line.strip()
        for key in ("traffic_bytes_per_launch:", "source_sha256_16:"):
            if line.startswith(key):
                vals[key] = line.split(":", 1)[1].strip()
    src = b"".join(open(os.path.join(ROOT, "paged_nvfp4_kv_gb300", "csrc", f), "rb").read()
                   for f in DECODE_SOURCES)
    if hashlib.sha256(src).hexdigest()[:16] != vals.get("source_sha256_16:"):
        return None
    return int(vals["traffic_bytes_per_launch:"])


def attention_flops(w):
    """QK^T + PV FLOPs of one step: every query row times its visible keys
    times head dim x 2 (multiply-add) x 2 (two products)."""
    tot = 0
    for b in range(w.batch):
        n, nq = int(w.seq_lens[b]), int(w.qlen[b])
        vis = (n - nq) * nq + nq * (nq + 1) // 2 if w.causal else n * nq
        tot += vis * w.num_q_heads
    return tot * w.head_dim * 4


def tensor_peak():
    """fp16/bf16 dense tensor peak in TFLOP/s (sustained figure: the tile
    kernel runs for most of a second)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        for key in ("bf16_tflops_sustained", "bf16_tflops"):
            if key in d:
                return float(d[key]), "measured"
    return 1700.0, "fallback"


def workload(cfg):
    from paged_nvfp4_kv_gb300 import workloads as W
    return W.WORKLOADS[cfg]()


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)

class OracleSampler:
    """The float64 oracle's paged attention on the host cores, over a sample
    of sequence 0's last n keys: the rope table, the roped keys and the
    encoded pool are built once (untimed); ``time()`` runs the attention of
    all of the sequence's query rows over the sample once."""

    def __init__(self, w):
        sys.path.insert(0, os.path.join(ROOT, "tests"))
        import oracle_path
        from oracle import attention as OA
        from oracle import paged as OP
        from oracle import yarn as OY
        self.w, self.OA, self.OP = w, OA, OP
        self.L = int(w.seq_lens[0])
        self.dtype = {"nvfp4": OP.NVFP4, "fp8": OP.FP8, "int8": OP.INT8, "bf16": OP.BF16}[w.kv_dtype]
        self.cos_t, self.sin_t = OY.rope_tables(w.yarn, self.L)
        self.q = oracle_path.roped_new_q(w, self.cos_t, self.sin_t)[: int(w.qlen[0])]
        self.OY = OY
        self.n = 0

    def prepare(self, n):
        w, OP = self.w, self.OP
        n = max(16, min(self.L, (n // 16) * 16))
        npg = (n + 15) // 16
        self.pool = OP.new_pool(npg, self.dtype, w.num_kv_heads, w.head_dim)
        self.table = np.arange(npg, dtype=np.int32)
        k = w.k_rows(0, self.L - n, self.L).astype(np.float64)
        v = w.v_rows(0, self.L - n, self.L).astype(np.float64)
        kr = self.OY.rope_rows(k, np.arange(self.L - n, self.L), self.cos_t, self.sin_t, w.yarn["rotary_dim"])
        OP.scatter_sequence_fast(self.pool, self.dtype, w.num_kv_heads, w.head_dim, self.table, 0, kr, v,
                                 w.g_k, w.g_v)
        self.n = n
        return n

    def time(self):
        w = self.w
        t0 = time.perf_counter()
        self.OA.paged_decode(self.pool, self.dtype, w.num_kv_heads, w.head_dim, self.q,
                             np.array([0, self.q.shape[0]]), self.table[None, :], np.array([self.n]),
                             w.num_q_heads, True, w.g_k, w.g_v)
        return time.perf_counter() - t0

    def calibrate(self, seconds, n0=4096):
        """Prepare a sample that takes about ``seconds`` per ``time()``."""
        self.prepare(n0)
        dt = self.time()
        return self.prepare(int(self.n * seconds / max(dt, 1e-4)))


def oracle_rate(w, seconds):
    """KV tokens/s/layer of the float64 oracle over a sample of sequence 0's
    keys sized to take about ``seconds``."""
    o = OracleSampler(w)
    n = o.calibrate(seconds)
    dt = o.time()
    return n / dt, n, dt


def cpu_info():
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return cores


def workload_config(w, world):
    """The ``config`` object of both arms' JSON lines."""
    return {"workload": w.name, "keys": int(w.seq_lens.sum()), "kv_dtype": w.kv_dtype,
            "query_rows": int(w.total_q) * w.num_q_heads, "heads": "24q/4kv x 256",
            "pages": int(w.num_pages), "l2": "inputs larger than L2 (no flush)",
            "parallelism": "replicas" if world > 1 else "single"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = workload(args.config)
    # each step is one oracle pass over a bounded sample, sized so the whole
    # run takes about two minutes of host time
    per_step = min(2.0, max(0.01, 120.0 / max(1, args.steps + args.warmup)))
    o = OracleSampler(w)
    keys = o.calibrate(per_step)
    times = []
    for i in range(args.warmup + args.steps):
        dt = o.time()
        if i >= args.warmup:
            times.append(dt)
    rate = keys / float(np.mean(times))
    cores = cpu_info()
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * float(np.mean(times)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d of %d keys of sequence 0, all %d query heads, per step"
                                   % (keys, int(w.seq_lens[0]), w.num_q_heads)},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# GPU arm

def l2_flusher(torch, nbytes=512 << 20):
    """A function that evicts L2 (129 MB on GB300) by writing a larger buffer."""
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    return lambda: buf.zero_()


def measure_steps(s, K, W, stream, local, flush=None, q_scale=None):
    """W warm-up steps, then K timed steps (append -> attention -> combine)
    with CUDA events on the launching stream, and a second pass with events
    between the three calls for per-kernel means.  With ``flush`` (inputs that
    fit in L2) each step is timed on its own after an L2 flush outside its
    events.  ``q_scale``: the FP4-query prefill instead of the bf16-query
    attention."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(W):
            s.step(q_scale=q_scale)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    with clocks:
        with torch.cuda.stream(stream):
            if flush is None:
                start = torch.cuda.Event(enable_timing=True)
                stop = torch.cuda.Event(enable_timing=True)
                start.record(stream)
                for _ in range(K):
                    s.step(q_scale=q_scale)
                stop.record(stream)
                stream.synchronize()
                step_ms = start.elapsed_time(stop) / K
            else:
                evs = []
                for _ in range(K):
                    flush()
                    e = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    e[0].record(stream)
                    s.step(q_scale=q_scale)
                    e[1].record(stream)
                    evs.append(e)
                stream.synchronize()
                step_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    with torch.cuda.stream(stream):
        for i in range(K):
            if flush is not None:
                flush()
            ev[i][0].record(stream)
            s.append()
            ev[i][1].record(stream)
            s.partials(q_scale)
            ev[i][2].record(stream)
            s.combine()
            ev[i][3].record(stream)
    stream.synchronize()
    return {"step_ms": step_ms,
            "append_ms": float(np.mean([e[0].elapsed_time(e[1]) for e in ev])),
            "decode_ms": float(np.mean([e[1].elapsed_time(e[2]) for e in ev])),
            "combine_ms": float(np.mean([e[2].elapsed_time(e[3]) for e in ev])),
            "clocks": clocks.summary(), "dev_err": s.error_word()}


def is_tile_path(w):
    return int(w.qlen.max()) * (w.num_q_heads // w.num_kv_heads) > 64


NOMINAL_FP4_OVER_BF16 = 13.5 / 2.25   # dense tensor rates of GB300, nominal


def roofline_of(w, decode_ms, fp4q=False):
    """Roofline of the step's dominant kernel: HBM bytes of KV + scales for
    the split-KV decode, causal-exact QK^T + PV FLOPs for the tensor-core tile.
    With NVFP4 queries half of the FLOPs (QK^T) run at the FP4 rate and half
    (P V) at the fp16 rate; the peak is then the harmonic combination of the
    two rates, the FP4 one taken as the measured bf16 peak times the nominal
    FP4 / bf16 ratio."""
    keys = int(w.seq_lens.sum())
    if is_tile_path(w):
        flops = attention_flops(w)
        tflops = flops / (decode_ms * 1e-3) / 1e12
        tpeak, tkind = tensor_peak()
        kernel = "prefill_tile_kernel (tcgen05, kind::f16)"
        if fp4q:
            tpeak = 2.0 / (1.0 / (tpeak * NOMINAL_FP4_OVER_BF16) + 1.0 / tpeak)
            tkind += " (QK^T at bf16 x 13.5/2.25, P V at bf16)"
            kernel = "prefill_tile_kernel (tcgen05, kind::mxf4nvf4 QK^T + kind::f16 P V)"
        return {"bound": "tensor", "achieved": tflops, "peak": tpeak, "unit": "TFLOP/s",
                "frac": tflops / tpeak, "traffic": None, "peak_kind": tkind,
                "kernel": kernel, "algorithmic_flops_per_launch": flops}
    peak, peak_kind = peaks()
    algo_bytes = keys * ALGO_BYTES_PER_TOKEN[w.kv_dtype]
    achieved = algo_bytes / (decode_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": profiled_traffic(w.kv_dtype) if keys == 1 << 20 else None,
            "peak_kind": peak_kind, "kernel": "paged_decode_attention",
            "algorithmic_bytes_per_launch": algo_bytes}


def config_record(cfg, K, W, local, fp4q=False):
    """One workload's step measured on its own (fill untimed): kernel times,
    the dominant kernel's roofline, the clock record of its timed region.
    ``fp4q``: the prefill chunk with NVFP4-encoded queries (block-scaled FP4
    QK^T, paged_prefill_attention_fp4q) instead of bf16 queries."""
    import torch
    from paged_nvfp4_kv_gb300.engine import DecodeSession
    w = workload(cfg)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        s = DecodeSession(w, device="cuda", stream=stream)
        s.fill()
    torch.cuda.synchronize()
    pool_bytes = s.cache.pool.numel()
    flush = l2_flusher(torch) if pool_bytes < (256 << 20) else None
    m = measure_steps(s, K, W, stream, local, flush, q_scale=w.g_q if fp4q else None)
    roof = roofline_of(w, m["decode_ms"], fp4q)
    keys = int(w.seq_lens.sum())
    rec = {"workload": w.name + (", NVFP4 queries (block-scaled FP4 QK^T)" if fp4q else ""),
           "kv_dtype": w.kv_dtype, "keys": keys,
           "query_rows": int(w.total_q) * w.num_q_heads, "steps": K, "warmup": W,
           "l2": "flushed before each step (pool fits in L2)" if flush else "pool larger than L2",
           "step_ms": m["step_ms"],
           "kernels_ms": {"kv_append_nvfp4": m["append_ms"], "paged_decode_attention": m["decode_ms"],
                          "split_kv_combine": m["combine_ms"]},
           "value": keys / (m["step_ms"] * 1e-3), "unit": UNIT,
           "roofline": {k: roof[k] for k in ("bound", "achieved", "peak", "unit", "frac", "peak_kind",
                                             "kernel")},
           "clocks": m["clocks"], "dev_err": m["dev_err"]}
    del s
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch
    import __graft_entry__
    __graft_entry__.build()
    from paged_nvfp4_kv_gb300.engine import DecodeSession

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    w = workload(args.config)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        s = DecodeSession(w, device="cuda", stream=stream)
        s.fill()
    torch.cuda.synchronize()

    K, W = args.steps, args.warmup
    qs = w.g_q if (args.fp4q and is_tile_path(w)) else None
    with torch.cuda.stream(stream):
        for _ in range(W):
            s.step(q_scale=qs)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    # the headline: K whole steps back to back, events only around the loop,
    # then the per-kernel pass (measure_steps; its warm-up is already done)
    m = measure_steps(s, K, 0, stream, local, q_scale=qs)
    if world > 1:
        dist.barrier()
    ms_per_step = replica_max(m["step_ms"], world, "cuda")
    keys = int(w.seq_lens.sum())
    value = replica_rate(keys, ms_per_step, world)

    # ---- end to end through the public API, host buffers
    qh = s.q.cpu().pin_memory()
    kh = s.k.cpu().pin_memory()
    vh = s.v.cpu().pin_memory()
    out_h = torch.empty(s.out.shape, dtype=s.out.dtype).pin_memory()
    h2d = qh.numel() * 2 + kh.numel() * 2 + vh.numel() * 2
    d2h = out_h.numel() * 2
    with torch.cuda.stream(stream):
        for _ in range(W):
            s.q.copy_(qh, non_blocking=True)
            s.k.copy_(kh, non_blocking=True)
            s.v.copy_(vh, non_blocking=True)
            s.step(q_scale=qs)
            out_h.copy_(s.out, non_blocking=True)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            s.q.copy_(qh, non_blocking=True)
            s.k.copy_(kh, non_blocking=True)
            s.v.copy_(vh, non_blocking=True)
            s.step(q_scale=qs)
            out_h.copy_(s.out, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e2e_ms = replica_max(e0.elapsed_time(e1) / K, world, "cuda")
    e2e_value = replica_rate(keys, e2e_ms, world)
    err = s.error_word()

    roofline = roofline_of(w, m["decode_ms"], qs is not None)
    tile_path = is_tile_path(w)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp16-mma/fp32-softmax over %s KV" % w.kv_dtype,
        "data": "synthetic",
        "config": dict(workload_config(w, world), **({"queries": "NVFP4 (block-scaled FP4 QK^T)"} if qs else {})),
        "kernels_ms": {"kv_append_nvfp4": m["append_ms"], "paged_decode_attention": m["decode_ms"],
                       "split_kv_combine": m["combine_ms"]},
        "hbm_gbs_decode": roofline["achieved"] if roofline["bound"] == "hbm" else None,
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        # per step: append, decode (plus its metadata kernel on the tile path), combine
        "gpu_launches": (4 if tile_path else 3) * K,
        "clocks": m["clocks"],
        "dev_err": err,
    }
    del s
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    if args.layers > 1:
        line["layers_graph"] = layer_stack_ms(w, args.layers, max(K, 50), max(W, 3))
    if not args.no_configs and world == 1:
        # every other workload, measured on its own after the headline
        recs = {}
        for cfg in (1, 2, 4, 5, 7, 8):
            if cfg == args.config:
                continue
            kc, wc = (3, 1) if cfg == 5 else (max(20, min(K, 200)), max(3, W))
            recs[str(cfg)] = config_record(cfg, kc, wc, local)
        recs["5-fp4q"] = config_record(5, 3, 1, local, fp4q=True)
        line["configs"] = recs
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, dt = oracle_rate(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cpu_info(), "kind": "oracle",
                                "sample": "%d of %d keys of sequence 0, all %d query heads"
                                          % (n, int(w.seq_lens[0]), w.num_q_heads),
                                "seconds": dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def layer_stack_ms(w, layers, K, W):
    """Per-token latency of ``layers`` attention layers (each its own pool,
    append -> decode -> combine) replayed from one CUDA graph; CUDA events
    around K replays after W warm-up replays.  The layers' pools start as
    byte copies of one filled pool (the same work per layer; per-layer
    contents are checked against the oracle by the graph tests)."""
    import torch
    from paged_nvfp4_kv_gb300.engine import DecodeStack
    st = DecodeStack.replicated(w, layers)
    st.fill()
    st.capture()
    for _ in range(W):
        st.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device())
    with clocks:
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(K):
            st.replay()
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / K
    err = st.error_word()
    del st
    torch.cuda.empty_cache()
    return {"layers": layers, "replays": K, "ms_per_token": ms, "ms_per_layer": ms / layers,
            "launches_per_replay": 3 * layers, "clocks": clocks.summary(), "dev_err": err}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Benchmark: one continuous-batching decode step of PagedAttention on GB300.

A step appends one new token per sequence to the paged KV cache (reshape_and_cache)
and runs paged_attention_decode over every sequence's full context.  The default
workload is the largest single-GPU one, the long-context split-K batch (8 sequences of
32768 tokens, 32/32 heads, head_dim 128, bf16 KV with one key channel scaled x8,
shuffled 1.25x block pool: 4.3 GB of K/V read per step); ``--workload`` names the others.

Printed: one JSON line (rank 0).  `value` is KV-read GB/s over the whole step
(algorithmic bytes: cached K/V actually attended + q + out + tables + the append),
inputs resident in HBM.  Inputs are larger than L2 (the pool is >1 GB), so no L2 flush
is done between steps.

The ``*_verify4`` workloads time a speculative-decoding verification step instead: 4
draft tokens per sequence are appended, then one multi-query call attends each draft
causally over the cache.  ``long_32k_window4k`` decodes the long_32k cache with a 4096-token
sliding window (bytes count the tokens each sequence's window covers).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                       [--workload NAME] [--seqs N]
``--seqs N`` keeps only the first N sequences of the workload (a smaller case of the same
shape, for profiler captures).
For N > 1 run under torch.distributed.run: each rank runs its own independent batch of
the same shape (weak scaling; the only collectives are the timing barrier and the
max-over-ranks reduction).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

from paged_kv_cache_264_gb300 import roofline, workloads as W  # noqa: E402

METRIC = "paged decode attention: KV-read GB/s (% of HBM peak) and decode steps/s"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "long_32k"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.txt")
CSRC = os.path.join(ROOT, "paged_kv_cache_264_gb300", "csrc")


KERNEL_SOURCES = {
    # sources that define each decode kernel family (a capture stays valid while they are unchanged)
    "cuda_core": ["pkv_device.cuh", "pkv_internal.h", "pkv_decode.cuh", "pkv_decode_bf16.cu",
                  "pkv_decode_int8.cu"],
    "tensor_core": ["pkv_device.cuh", "pkv_internal.h", "pkv_decode.cuh", "pkv_decode_mma.cuh",
                    "pkv_decode_mma.cu", "pkv_decode_mma_bf16.cu", "pkv_decode_mma_int8.cu",
                    "pkv_decode_mma_fp8.cu", "pkv_decode_mma_quant_d64.cu"],
}


def _code_only(text: str) -> str:
    """Source text without comments and whitespace: a capture stays valid across comment edits."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return re.sub(r"\s+", "", text)


def kernel_source_hash(kernel: str = "cuda_core") -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes of the decode kernel from a committed ncu capture, if it was
    taken on the current sources of that kernel."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    current = kernel_source_hash(kernel)
    with open(TRAFFIC_FILE) as f:
        for line in f:
            if line.startswith("#") or "=" not in line:
                continue
            rec = dict(kv.split("=", 1) for kv in line.split())
            if (rec.get("workload") == workload and rec.get("kernel") == kernel
                    and rec.get("source_hash") == current):
                return int(rec["dram_bytes"])
    return None


# ------------------------------------------------------------------ distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------------------ our arm

def make_workload(name: str, seqs: int, device):
    """The named workload, or a batch of its first ``seqs`` sequences' lengths with the
    same head shape, pool type and value distribution, in a shuffled pool sized 1.25x what
    those sequences need (a smaller case of the same shape: device memory shrinks with it)."""
    if not seqs:
        return W.make(name, device=device)
    spec = W.SPECS[name]
    if not 1 <= seqs <= spec.num_seqs:
        raise SystemExit(f"--seqs must be in 1..{spec.num_seqs}")
    lens = W.context_lens_of(name)[:seqs]
    return W.build(name=name, context_lens=lens, num_q_heads=spec.num_q_heads,
                   num_kv_heads=spec.num_kv_heads, head_dim=spec.head_dim, kv_dtype=spec.kv_dtype,
                   seed=spec.seed,
                   outlier_key_channel_frac=spec.outlier_key_channel_frac,
                   outlier_key_scale=spec.outlier_key_scale, device=device,
                   num_queries=spec.num_queries)


def run_ours(args, rank, world, local):
    import paged_kv_cache_264_gb300 as pkv
    from paged_kv_cache_264_gb300 import build as pkv_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (there is no CPU path)")
    pkv_build.build()
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    spec = W.SPECS[args.workload]
    w = make_workload(args.workload, args.seqs, dev)
    kv = spec.kv_dtype
    stream = torch.cuda.current_stream(dev)

    pool = pkv.PagedKVPool(w.num_blocks, w.num_kv_heads, w.head_dim, kv, device=dev, fill=0)
    hist, last = w.history_rows().to(dev), w.last_token_rows().to(dev)
    slots = w.slot_mapping.to(dev)
    if hist.numel():
        pool.reshape_and_cache(w.key[hist].contiguous(), w.value[hist].contiguous(), slots[hist].contiguous())
    new_k, new_v = w.key[last].contiguous(), w.value[last].contiguous()
    new_slots = slots[last].contiguous()
    w.key = w.value = None  # the history now lives in the pool; keep only the step's rows
    del hist, slots
    torch.cuda.empty_cache()
    q = w.q.to(dev)
    tables = w.block_tables.to(dev)
    lens = w.context_lens.to(dev)
    out = torch.empty_like(q)
    max_ctx = w.max_context_len
    nq, win = w.num_queries, spec.window
    kern = args.kernel
    ws_n = pkv.decode_workspace_bytes(pool, w.num_seqs, w.num_q_heads, max_ctx, kernel=kern, num_queries=nq,
                                      window=win)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    plan = pkv.decode_plan(pool, w.num_seqs, w.num_q_heads, max_ctx, kernel=kern, num_queries=nq, window=win)
    torch.cuda.synchronize(dev)
    assert pool.device_error() == 0

    def step():
        pkv.reshape_and_cache(pool, new_k, new_v, new_slots, stream)
        pkv.paged_attention_decode(pool, q, tables, lens, w.scale, max_ctx, out=out, workspace=ws,
                                   kernel=kern, window=win, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    def decode():
        pkv.paged_attention_decode(pool, q, tables, lens, w.scale, max_ctx, out=out, workspace=ws,
                                   kernel=kern, window=win, stream=stream)

    # ---- timed region: K steps between one pair of CUDA events.  A CUDA event recorded
    # between two launches keeps the programmatic dependent launch from overlapping them
    # (about 4 us per event pair here), so the decode call's own timing is taken in the two
    # decode loops after it, inside the same clock-sampled span.
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index if world == 1 else local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    launches0 = pkv.launch_count()
    t0.record(stream)
    for i in range(args.steps):
        pkv.reshape_and_cache(pool, new_k, new_v, new_slots, stream)
        decode()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    launches = pkv.launch_count() - launches0
    # the decode call: K calls back to back between one event pair (its mean), then K calls
    # each between its own pair of events (the distribution; each includes an event's cost)
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    for i in range(args.steps):
        decode()
    d1.record(stream)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record(stream)
        decode()
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    ms_total = t0.elapsed_time(t1)
    ms_total = max_over_ranks(ms_total, world, dev)
    dec_ms = max_over_ranks(d0.elapsed_time(d1), world, dev) / args.steps
    dec_all = sorted(a.elapsed_time(b) for a, b in ev)
    dec_ev_mean = sum(dec_all) / args.steps
    dec_median = statistics.median(dec_all)
    dec_p90 = dec_all[min(len(dec_all) - 1, math.ceil(0.9 * len(dec_all)) - 1)]
    assert pool.device_error() == 0

    sb = roofline.step_bytes(w.context_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, kv,
                             num_queries=nq, window=win)
    ms_step = ms_total / args.steps
    total_bytes = sum_over_ranks(float(sb.step) * args.steps, world, dev)
    value = total_bytes / (ms_total * 1e-3) / 1e9
    steps_per_s = args.steps * world / (ms_total * 1e-3)

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, pkv, pool, w, new_k, new_v, new_slots, q, tables, lens, max_ctx, ws, sb,
                  stream, dev, world, win, kern, out_ref=out)

    peak, peak_kind = measured_peaks()
    achieved = sb.decode / (dec_ms * 1e-3) / 1e9
    traffic = None if args.seqs else recorded_traffic(args.workload, plan["kernel"])
    kernel = ("paged_decode_mma_kernel" if plan["kernel"] == "tensor_core" else "paged_decode_kernel") + (
        " + lse_reduce_kernel" if plan["kernels_per_call"] == 2 else "")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "int8": "int8 KV, fp32 accumulate", "fp8": "fp8 e4m3 KV, fp32 accumulate"}[kv],
        "data": "synthetic (seeded N(0,1) bf16 values; seeded lengths and shuffled block pool)",
        "config": {
            "workload": args.workload, "description": spec.description,
            "subset": f"first {args.seqs} of {spec.num_seqs} sequences" if args.seqs else None,
            "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads, "num_kv_heads": w.num_kv_heads,
            "head_dim": w.head_dim, "kv_dtype": kv, "sum_context_tokens": int(w.context_lens.sum()),
            "max_context_len": max_ctx, "num_blocks": w.num_blocks,
            "step": ("reshape_and_cache of one new token per sequence + paged_attention_decode" if nq == 1 else
                     f"reshape_and_cache of {nq} draft tokens per sequence + one multi-query "
                     f"paged_attention_decode verifying them (causal over the last {nq} positions)"),
            "num_queries": nq, "window": win or None, "kernel_option": kern,
            "plan": plan, "l2": "inputs larger than L2 (pool %.2f GB > 129 MB); no flush" % (
                2 * pool.k_cache.numel() * pool.k_cache.element_size() / 1e9),
            "parallelism": f"{world} independent replicas" if world > 1 else "single GPU",
        },
        "decode_steps_per_s": round(steps_per_s, 1),
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "bytes_per_step": sb.step,
        "roofline": {
            "kernel": kernel, "bound": "hbm", "achieved": round(achieved, 2),
            "peak": peak, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
            "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
            "algorithmic_bytes_per_launch": sb.decode, "avg_launch_ms": round(dec_ms, 5),
            "launch_timing": ("avg_launch_ms: K decode calls back to back between one pair of CUDA events "
                              "on the launching stream; *_evented: K calls each between its own pair "
                              "(an event between launches stops the programmatic dependent launch "
                              "from overlapping them)"),
            "avg_launch_ms_evented": round(dec_ev_mean, 5),
            "median_launch_ms": round(dec_median, 5), "p90_launch_ms": round(dec_p90, 5),
            "frac_median": round(sb.decode / (dec_median * 1e-3) / 1e9 / peak, 4),
            "launches_timed": len(dec_all),
        },
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    pool.close()
    return line


def run_e2e(args, pkv, pool, w, new_k, new_v, new_slots, q, tables, lens, max_ctx, ws, sb, stream,
            dev, world, win=0, kern="auto", out_ref=None):
    """Same step through the public API, but every step copies its inputs from pinned
    host memory and reads the output back.  The step's inputs (q, the appended K/V rows,
    their slots, the page tables and lengths) sit in one pinned staging buffer and go to
    the device in one copy; the output comes back in one copy.

    Reported twice: ``value`` with the copies double-buffered (two device input buffers and
    two outputs; step i + 1's inputs travel on an upload stream and step i's output on a
    download stream while step i computes, as a serving loop would run it), and
    ``serial_value`` with upload, compute and download in order on one stream.  Either way
    every step moves all of its bytes, and the last output read back must equal the device
    path's output bit for bit."""
    parts = [("q", q), ("k", new_k), ("v", new_v), ("slots", new_slots), ("tables", tables), ("lens", lens)]
    offs, size = {}, 0
    for name, t in parts:
        nbytes = t.numel() * t.element_size()
        offs[name] = (size, nbytes)
        size += (nbytes + 255) // 256 * 256  # 256-byte aligned views
    host_buf = torch.empty(size, dtype=torch.uint8).pin_memory()
    for name, t in parts:
        o, nbytes = offs[name]
        host_buf[o:o + nbytes].copy_(t.contiguous().cpu().view(torch.uint8).reshape(-1))
    dev_buf = [torch.empty(size, dtype=torch.uint8, device=dev) for _ in range(2)]
    dbuf = [{name: dev_buf[j][o:o + nb].view(t.dtype).view(t.shape)
             for (name, t), (o, nb) in zip(parts, (offs[n] for n, _ in parts))} for j in range(2)]
    out_d = [torch.empty_like(q) for _ in range(2)]
    out_h = [torch.empty(q.shape, dtype=q.dtype).pin_memory() for _ in range(2)]
    h2d = size
    d2h = out_h[0].numel() * out_h[0].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_back = [torch.cuda.Event() for _ in range(2)]

    def compute(j):
        d = dbuf[j]
        pkv.reshape_and_cache(pool, d["k"], d["v"], d["slots"], stream)
        pkv.paged_attention_decode(pool, d["q"], d["tables"], d["lens"], w.scale, max_ctx,
                                   out=out_d[j], workspace=ws, kernel=kern, window=win, stream=stream)

    def step_serial(i):
        dev_buf[0].copy_(host_buf, non_blocking=True)
        compute(0)
        out_h[0].copy_(out_d[0], non_blocking=True)

    def step_overlap(i):
        j = i % 2
        with torch.cuda.stream(up):
            up.wait_event(done[j])  # step i - 2 has consumed this input buffer
            dev_buf[j].copy_(host_buf, non_blocking=True)
            in_ready[j].record(up)
        stream.wait_event(in_ready[j])
        stream.wait_event(out_back[j])  # step i - 2's output has left this buffer
        compute(j)
        done[j].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(done[j])
            out_h[j].copy_(out_d[j], non_blocking=True)
            out_back[j].record(down)

    def timed(step, n):
        for i in range(max(3, args.warmup)):
            step(i)
        torch.cuda.synchronize(dev)
        barrier(world)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        up.wait_event(a)
        down.wait_event(a)
        for i in range(n):
            step(i)
        if step is step_overlap:
            stream.wait_event(out_back[(n - 1) % 2])  # the last output is back on the host
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        return max_over_ranks(a.elapsed_time(b), world, dev)

    n = max(10, min(args.steps, 500))
    ms_serial = timed(step_serial, n)
    if out_ref is not None and not torch.equal(out_h[0], out_ref.cpu()):
        raise RuntimeError("the serial end-to-end output differs from the device path's")
    ms = timed(step_overlap, n)
    if out_ref is not None and not torch.equal(out_h[(n - 1) % 2], out_ref.cpu()):
        raise RuntimeError("the double-buffered end-to-end output differs from the device path's")
    total = sum_over_ranks(float(sb.step) * n, world, dev)
    return {"value": round(total / (ms * 1e-3) / 1e9, 2), "unit": UNIT, "steps": n,
            "ms_per_step": round(ms / n, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies": "double-buffered on upload/download streams",
            "serial_value": round(total / (ms_serial * 1e-3) / 1e9, 2),
            "serial_ms_per_step": round(ms_serial / n, 5)}


# ------------------------------------------------------------------ oracle legs

def oracle_sample(workload: str, target_s: float):
    """A bounded sample of the workload for the CPU oracle: the first k sequences (values
    regenerated on the host), their blocks compacted into an oracle-side pool, the append
    rows, and the algorithmic bytes of that sample's step."""
    import numpy as np

    import oracle

    o = oracle.load()
    spec = W.SPECS[workload]
    lens_all = W.context_lens_of(workload)
    order = list(range(spec.num_seqs))

    def build(k):
        w = W.make(workload, seqs=order[:k])
        shape_tok = w.num_tokens
        nblk = (w.context_lens.numpy() + 15) // 16
        nb = int(nblk.sum())
        tab = np.full((k, int(nblk.max())), -1, np.int32)
        c = 0
        for i, n in enumerate(nblk):
            tab[i, :n] = np.arange(c, c + n)
            c += n
        lens = w.context_lens.numpy().astype(np.int32)
        slots = np.empty(shape_tok, np.int32)
        for i in range(k):
            lo = int(w.seq_offsets[i])
            t = np.arange(int(lens[i]))
            slots[lo:lo + lens[i]] = tab[i, t // 16] * 16 + t % 16
        shape = (nb, w.num_kv_heads, 16, w.head_dim)
        key, value = W.bf16_bits(w.key), W.bf16_bits(w.value)
        hist, last = w.history_rows().numpy(), w.last_token_rows().numpy()
        if spec.kv_dtype == "bf16":
            pool = dict(k_cache=np.zeros(shape, np.uint16), v_cache=np.zeros(shape, np.uint16))
            o.reshape_and_cache_bf16(key[hist], value[hist], slots[hist], pool["k_cache"], pool["v_cache"])
        else:
            cdt = np.int8 if spec.kv_dtype == "int8" else np.uint8
            pool = dict(k_cache=np.zeros(shape, cdt), v_cache=np.zeros(shape, cdt),
                        k_scale=np.zeros(shape[:3], np.float32), v_scale=np.zeros(shape[:3], np.float32))
            write_q(key[hist], value[hist], slots[hist], pool["k_cache"], pool["v_cache"],
                    pool["k_scale"], pool["v_scale"])
        args = dict(q=W.bf16_bits(w.q), key=key[last], value=value[last], slots=slots[last], tab=tab,
                    lens=lens, scale=w.scale)
        sb = roofline.step_bytes(w.context_lens, w.num_q_heads, w.num_kv_heads, w.head_dim, spec.kv_dtype,
                                 num_queries=spec.num_queries, window=spec.window)
        if spec.num_queries == 1 and spec.window:
            args["q"] = args["q"][:, None]  # one query token, through the windowed decode
        return pool, args, sb

    write_q = o.reshape_and_cache_int8 if spec.kv_dtype == "int8" else o.reshape_and_cache_fp8
    if spec.window:
        decode = lambda *a: o.paged_decode_multi(*a, window=spec.window)
    else:
        decode = o.paged_decode_multi if spec.num_queries > 1 else o.paged_decode

    def run(pool, a):
        if spec.kv_dtype == "bf16":
            o.reshape_and_cache_bf16(a["key"], a["value"], a["slots"], pool["k_cache"], pool["v_cache"])
            decode(a["q"], pool["k_cache"], pool["v_cache"], a["tab"], a["lens"], a["scale"])
        else:
            write_q(a["key"], a["value"], a["slots"], pool["k_cache"], pool["v_cache"],
                    pool["k_scale"], pool["v_scale"])
            decode(a["q"], pool["k_cache"], pool["v_cache"], a["tab"], a["lens"], a["scale"],
                   pool["k_scale"], pool["v_scale"])

    # calibrate on one sequence, then size the sample to about target_s per step
    pool, a, sb = build(1)
    t = time.perf_counter()
    run(pool, a)
    per_token = (time.perf_counter() - t) / max(1, int(lens_all[0]))
    k, tokens = 0, 0
    while k < spec.num_seqs and (tokens + int(lens_all[k])) * per_token <= target_s:
        tokens += int(lens_all[k])
        k += 1
    k = max(k, 1)
    pool, a, sb = build(k)
    return o, pool, a, sb, run, k


def cpu_baseline(workload: str, seconds: float):
    o, pool, a, sb, run, k = oracle_sample(workload, seconds)
    t = time.perf_counter()
    n = 0
    while True:
        run(pool, a)
        n += 1
        if time.perf_counter() - t >= seconds * 0.5:
            break
    dt = (time.perf_counter() - t) / n
    return {"value": round(sb.step / dt / 1e9, 4), "unit": UNIT, "cores": o.max_threads(),
            "kind": "oracle",
            "sample": f"first {k} of {W.SPECS[workload].num_seqs} sequences, full step (append + decode), "
                      f"{n} repetition(s), {dt:.3f} s each, fp64 C oracle with OpenMP"}


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, unchanged, on a bounded sample per step."""
    if rank != 0:
        return None
    budget = 120.0
    per_step = max(0.02, budget / max(1, args.steps + args.warmup))
    o, pool, a, sb, run, k = oracle_sample(args.workload, per_step)
    for _ in range(args.warmup):
        run(pool, a)
    t = time.perf_counter()
    for _ in range(args.steps):
        run(pool, a)
    dt = time.perf_counter() - t
    value = sb.step * args.steps / dt / 1e9
    spec = W.SPECS[args.workload]
    sample = (f"first {k} of {spec.num_seqs} sequences per step (append + decode), "
              f"fp64 C oracle with OpenMP")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": {"workload": args.workload, "description": spec.description},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": o.max_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(W.SPECS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work for the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--kernel", choices=["auto", "cuda_core", "tensor_core"], default="auto",
                    help="decode kernel family (auto: the plan's choice)")
    ap.add_argument("--seqs", type=int, default=0,
                    help="keep only the first N sequences (a smaller case for profiler captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1 and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Paged decode attention benchmark on GB300.

One step = one pass of the hot path over one batch of the bench workload:
append each request's newest K/V (pa_reshape_and_cache) then paged decode
attention over every request's context (pa_decode: split-K partitions and
the log-sum-exp merge).  Default workload ``c2``: bf16 MHA, 32 heads, head_dim
128, block_size 16, batch 64, context lengths U[128, 2048], a randomly
permuted 1.45 GB pool (larger than the 129 MB L2, so K/V stream from HBM).

Prints one JSON line.  ``value`` is HBM GB/s of algorithmic bytes (K/V rows
of every token in context, Q, O, the block-table entries and lengths, plus
the append's K/V rows read and written) over the device-timed K steps;
``seq_steps_per_s`` = batch / step time.  ``--impl reference`` times the
float64 CPU oracle on host cores on bounded samples of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
METRIC = "paged decode attention HBM GB/s (% of GB300 peak); seq-steps/s at batch 64"
WORKLOAD_TEXT = {
    "c2": "bf16 MHA decode: 32 heads, head_dim 128, block_size 16, batch 64, context U[128,2048], "
          "scattered pool; plus reshape_and_cache of 64 new tokens",
    "c3": "bf16 MHA decode: 40 heads, head_dim 128, block_size 16, batch 128, context log-normal "
          "(median 512, cap 4096), scattered pool; plus reshape_and_cache of 128 new tokens",
    "c4": "bf16 GQA decode: 32/8 heads, head_dim 128, block_size 16, batch 256, context U[1024,32768], "
          "split-K over 2048-token partitions (automatic); plus reshape_and_cache of 256 new tokens",
    "c4b32": "as c4 with block_size 32",
    "c2fp8": "as c2 over an e4m3 K/V pool with per-token fp32 scales (codes + scales read per token); "
             "append quantises the 64 new tokens",
    "c4fp8": "as c4 over an e4m3 K/V pool with per-token fp32 scales; append quantises the 256 new tokens",
    "swap": "preemption swap of the c2 pool layout (bf16, 32 heads, head_dim 128, block_size 16): "
            "4096 scattered blocks (1.07 GB of K+V) out to page-locked host memory and back into "
            "other scattered device blocks",
    "c5prefill": "bf16 GQA 32/8 causal chunked-prefill tile: 64 prompts, 512 queries at positions 512..1023 "
                 "over a 1024-token paged context (block_size 16), tensor cores",
    "mixed": "one mixed round in one launch (pa_prefill_varlen): 8 prompts each running a 512-token prefill "
             "chunk at the end of a 1024-token context + 256 decode requests over contexts U[128,2048]; "
             "bf16 GQA 32/8, head_dim 128, block_size 16",
    "c5": "bf16 GQA decode 32/8, 64 prompts x 8 samples sharing 1024-token prompts + private tails U[0,256] "
          "(pa_decode_shared: each shared block read once per prompt; GB/s counts each physical block once); "
          "plus reshape_and_cache of the new tokens",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="c2", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--long-repeat", type=int, default=2000,
                    help="decode legs: steps of the event-free repeat after a shorter timed region (0: none)")
    ap.add_argument("--no-share", action="store_true",
                    help="c5: run plain pa_decode instead of the shared-prefix path")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    return ap.parse_args()


def max_over_ranks(x, world, device):
    """The largest value of x over all ranks (the slowest rank's time); x
    itself for one rank.  Works with any process-group backend."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, total_ms, steps, world):
    """Whole-job throughput: the units all ranks processed (each rank runs the
    same workload on its own replica) over the slowest rank's time."""
    return world * units_per_rank / (total_ms / 1e3 / steps)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_hash(paths):
    """sha256 over the decode kernel's source files, in order."""
    h = hashlib.sha256()
    for p in paths:
        h.update(open(p, "rb").read())
    return h.hexdigest()


def _csrc(*names):
    return [os.path.join(ROOT, "paged_kv_cache_307_gb300", "csrc", f) for f in names]


DECODE_SOURCES = _csrc("pa_decode_kernel.cuh", "pa_decode.cu", "pa_mma.cuh", "pa_common.cuh")
FP8_SOURCES = _csrc("pa_decode_kernel.cuh", "pa_decode.cu", "pa_decode_fp8.cu", "pa_mma.cuh", "pa_common.cuh")
SHARED_SOURCES = _csrc("pa_decode_shared.cu", "pa_mma.cuh", "pa_common.cuh")


def traffic_record(workload, batch, sources=DECODE_SOURCES):
    """ncu DRAM bytes per launch of the decode kernel for the full-size bench
    workload, from a committed profile summary (captured at a smaller batch and
    scaled by algorithmic bytes where the summary says so); None if it is
    missing, is for another batch, or the kernel sources changed since."""
    p = os.path.join(ROOT, "profiles", "decode_%s_traffic.json" % workload)
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("batch") != batch or d.get("kernel_sha256") != kernel_hash(sources):
        return None
    return d.get("traffic_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 20 ms from just
    before the timed region until after it; the summary keeps the samples
    whose timestamps fall inside the region (begin() .. end()), or, for a
    region shorter than the sampling interval, the samples nearest to it."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.lines = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.Q, "--format=csv,noheader,nounits",
                                          "-lms", "20", "-i", str(self.index)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def begin(self):
        self.t0 = time.time()

    def end(self):
        self.t1 = time.time()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"error": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        import datetime
        rows = []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                ts = None
            try:
                rows.append((ts, float(f[2]), float(f[3]),
                             [n for n, val in zip(names, f[6:10]) if val.lower() == "active"]))
            except ValueError:
                continue
        if not rows:
            return {"error": "no samples"}
        sel, where = rows, "all samples (no region marks)"
        if self.t0 is not None and self.t1 is not None and all(r[0] is not None for r in rows):
            inside = [r for r in rows if self.t0 - 0.005 <= r[0] <= self.t1 + 0.005]
            if inside:
                sel, where = inside, "inside the timed region"
            else:
                mid = 0.5 * (self.t0 + self.t1)
                near = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
                sel, where = near, "nearest to the timed region (shorter than the 20 ms sampling interval)"
        reasons = sorted({n for r in sel for n in r[3]})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel), "which": where,
                "region_ms": round((self.t1 - self.t0) * 1e3, 2) if self.t0 and self.t1 else None}


def pipelined_e2e(stream, host_inputs, out_like, compute, n, warm=3):
    """End-to-end steps through the public API: every step uploads its inputs
    (pinned host tensors) and reads its result back, double-buffered so that
    step k+1's upload and step k-1's read-back (each on its own copy stream,
    so the two directions can run at once) overlap step k's compute.  ``compute(dev_inputs, out)`` enqueues one step on
    ``stream``.  Returns (ms for n steps, last result on the host, bytes
    uploaded per step, bytes read back per step)."""
    import torch
    devb = [{k: torch.empty_like(v, device=out_like.device) for k, v in host_inputs.items()} for _ in range(2)]
    outs = [torch.empty_like(out_like) for _ in range(2)]
    out_host = [torch.empty(out_like.shape, dtype=out_like.dtype).pin_memory() for _ in range(2)]
    up_stream = torch.cuda.Stream(device=out_like.device)
    down_stream = torch.cuda.Stream(device=out_like.device)
    ev_down = [torch.cuda.Event() for _ in range(2)]
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]

    def upload(k):
        i = k % 2
        with torch.cuda.stream(up_stream):
            if k >= 2:
                up_stream.wait_event(ev_done[i])        # buffers i are free again
            for name, t in host_inputs.items():
                devb[i][name].copy_(t, non_blocking=True)
            ev_up[i].record(up_stream)

    def step(k):
        i = k % 2
        stream.wait_event(ev_up[i])
        if k >= 2:
            stream.wait_event(ev_down[i])               # outs[i] has been read back
        compute(devb[i], outs[i])
        ev_done[i].record(stream)

    def download(k):
        i = k % 2
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(ev_done[i])
            out_host[i].copy_(outs[i], non_blocking=True)
            ev_down[i].record(down_stream)

    def run(m):
        upload(0)
        for k in range(m):
            if k + 1 < m:
                upload(k + 1)
            step(k)
            if k >= 1:
                download(k - 1)
        download(m - 1)
        stream.wait_stream(up_stream)
        stream.wait_stream(down_stream)

    run(warm)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(n)
    b.record(stream)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in host_inputs.values())
    d2h = out_host[0].numel() * out_host[0].element_size()
    return a.elapsed_time(b), out_host[(n - 1) % 2], h2d, d2h


# ---------------------------------------------------------------- CPU oracle legs

def _widen(u16):
    import numpy as np
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _oracle_slice(task):
    """One (sequence, KV head) slice through the oracle: append the newest
    token's K/V, then decode the query heads that read this KV head."""
    import numpy as np
    import oracle
    q, k, v, L, key, val, slot, scale = task
    k, v = oracle.reshape_and_cache(_widen(key)[None], _widen(val)[None], np.array([slot]),
                                    _widen(k), _widen(v))
    table = np.arange(k.shape[0])[None]
    return oracle.paged_decode(_widen(q)[None], k, v, table, np.array([L]), scale)


def _oracle_seq_fp8(task):
    """One sequence of an e4m3 workload through the oracle: quantise-append
    the newest token (all heads: the scale is per token), then decode."""
    import numpy as np
    import oracle
    q, kc, vc, ks, vs, L, key, val, slot, scale = task
    kc, vc, ks, vs = oracle.reshape_and_cache_fp8(_widen(key)[None], _widen(val)[None], np.array([slot]),
                                                  kc, vc, ks, vs)
    table = np.arange(kc.shape[0])[None]
    return oracle.paged_decode_fp8(_widen(q)[None], kc, vc, ks, vs, table, np.array([L]), scale)


def _cpu_tasks_fp8(name, nseq, seed):
    """Per-sequence oracle inputs of an e4m3 workload (compact pools of
    codes and scales), with their algorithmic bytes."""
    import numpy as np
    import torch
    from paged_kv_cache_307_gb300 import workloads as W
    c = W.fp8_case(W.decode_case(name[:-3], device="cpu", nan_fill=False, seed=seed, B=nseq))
    s = c.spec
    bs = s.bs
    lens, tables = c.context_lens.numpy(), c.block_tables.numpy()
    u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    tasks, nbytes = [], []
    for b in range(len(lens)):
        n = -(-int(lens[b]) // bs)
        blocks = tables[b, :n]
        slot = int(c.slot_mapping[b])
        local_slot = int(np.where(blocks == slot // bs)[0][0]) * bs + slot % bs
        tasks.append((u16(c.q[b]), c.k_cache[blocks].numpy(), c.v_cache[blocks].numpy(),
                      c.extra["k_scale"][blocks].numpy(), c.extra["v_scale"][blocks].numpy(), int(lens[b]),
                      u16(c.key[b]), u16(c.value[b]), local_slot, c.scale))
        nbytes.append(int(lens[b]) * (2 * s.Hkv * s.D + 8) + 2 * s.Hq * s.D * 2 + 4 * n + 4 + 8
                      + 2 * (s.Hkv * s.D * 2 + s.Hkv * s.D + 4))
    return tasks, nbytes


def _cpu_tasks(name, nseq, seed):
    """Oracle inputs per (sequence, KV head) slice, as bf16 bit patterns with
    the slice's blocks gathered into a compact pool, drawn by the same
    workload generator on the CPU.  Returns the tasks and their algorithmic
    bytes (the same accounting as the GPU leg)."""
    import numpy as np
    import torch
    from paged_kv_cache_307_gb300 import workloads as W
    c = W.decode_case(name, device="cpu", nan_fill=False, seed=seed, B=nseq)
    s = c.spec
    bs, G = s.bs, s.Hq // s.Hkv
    lens = c.context_lens.numpy()
    tables = c.block_tables.numpy()
    u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    kb, vb, qb, keyb, valb = u16(c.k_cache), u16(c.v_cache), u16(c.q), u16(c.key), u16(c.value)
    tasks, nbytes = [], []
    e = 2
    for b in range(len(lens)):
        n = -(-int(lens[b]) // bs)
        blocks = tables[b, :n]
        slot = int(c.slot_mapping[b])
        local_slot = int(np.where(blocks == slot // bs)[0][0]) * bs + slot % bs
        for g in range(s.Hkv):
            tasks.append((qb[b, g * G:(g + 1) * G], kb[blocks][:, :, g:g + 1].copy(),
                          vb[blocks][:, :, g:g + 1].copy(), int(lens[b]), keyb[b, g:g + 1],
                          valb[b, g:g + 1], local_slot, c.scale))
            nbytes.append(int(lens[b]) * 2 * s.D * e + 2 * G * s.D * e + (4 * n + 4 + 8) / s.Hkv
                          + 2 * 2 * s.D * e)
    return tasks, nbytes


def _pool(cores):
    import multiprocessing as mp
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[v] = "1"
    return mp.get_context("spawn").Pool(cores)


def cpu_baseline(name, seconds):
    """The oracle as it stands on (sequence, KV head) slices of a 16-sequence
    sample, spread over the host cores (spawn pool, one BLAS thread each),
    repeated until about `seconds` of wall time."""
    cores = os.cpu_count() or 1
    nseq = 16
    fp8 = name.endswith("fp8")
    tasks, nbytes = (_cpu_tasks_fp8 if fp8 else _cpu_tasks)(name, nseq, seed=12345)
    fn = _oracle_seq_fp8 if fp8 else _oracle_slice
    with _pool(cores) as pool:
        pool.map(fn, tasks[:cores])                     # worker start-up outside the timing
        t0 = time.perf_counter()
        reps = 0
        while True:
            pool.map(fn, tasks, chunksize=1 if fp8 else 4)
            reps += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
    gbs = reps * sum(nbytes) / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": "%d passes over a %d-sequence sample of workload %s, split into %d %s "
                      "slices (append + decode, float64), %.1f s wall"
                      % (reps, nseq, name, len(tasks), "sequence" if fp8 else "(sequence, KV head)", dt),
            "seq_steps_per_s": round(reps * nseq / dt, 3)}


def run_reference_prefill(args):
    """Oracle prefill on one host core: each step is a slice of the c5 tile
    (one prompt, 8 query rows at the end of its 1024-token context)."""
    import numpy as np
    import torch
    import oracle
    from paged_kv_cache_307_gb300 import workloads as W
    c = W.prefill_case(device="cpu", prompts=1, Tq=8, nan_fill=False)
    f64 = lambda t: t.to(torch.float64).numpy()
    k, v, q = f64(c["k_cache"]), f64(c["v_cache"]), f64(c["q"])
    tables, lens = c["block_tables"].numpy(), c["context_lens"].numpy()
    flops = W.prefill_flops(lens, 8, q.shape[2], q.shape[3])
    for _ in range(args.warmup):
        oracle.paged_prefill(q, k, v, tables, lens, c["scale"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_prefill(q, k, v, tables, lens, c["scale"])
    dt = time.perf_counter() - t0
    val = flops * args.steps / dt / 1e12
    line = {"impl": "reference", "metric": "chunked-prefill tile TFLOP/s (bf16, causal, unmasked work)",
            "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "c5prefill: " + WORKLOAD_TEXT["c5prefill"],
                       "sample": "one prompt, 8 query rows per step"},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": "%d steps of 8 query rows x 32 heads over a 1024-token context" % args.steps},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _swap_sample(nblk, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    shape = (nblk, 16, 32, 128)
    k = rng.integers(0, 1 << 16, size=(2 * nblk,) + shape[1:], dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(2 * nblk,) + shape[1:], dtype=np.uint16)
    hk, hv = np.zeros(shape, np.uint16), np.zeros(shape, np.uint16)
    perm = rng.permutation(2 * nblk)
    out_pairs = np.stack([perm[:nblk], np.arange(nblk)], 1)
    in_pairs = np.stack([np.arange(nblk), perm[nblk:]], 1)
    return k, v, hk, hv, out_pairs, in_pairs


def swap_cpu_once(sample):
    import oracle
    k, v, hk, hv, out_pairs, in_pairs = sample
    hk, hv = oracle.swap_blocks(hk, hv, k, v, out_pairs)
    return oracle.swap_blocks(k, v, hk, hv, in_pairs)


def run_reference_swap(args):
    """Oracle swap on one host core: each step swaps a 64-block sample of the
    swap workload out and back in (the oracle copies whole pools)."""
    sample = _swap_sample(64, 5)
    moved = 2 * 2 * 64 * 16 * 32 * 128 * 2
    for _ in range(args.warmup):
        swap_cpu_once(sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        swap_cpu_once(sample)
    dt = time.perf_counter() - t0
    val = moved * args.steps / dt / 1e9
    line = {"impl": "reference", "metric": "KV block swap GB/s (device <-> page-locked host, both directions)",
            "value": round(val, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "u16", "data": "synthetic",
            "config": {"workload": "swap: " + WORKLOAD_TEXT["swap"], "sample": "64 blocks out and back per step"},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": "%d steps of 64 blocks out and back" % args.steps},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_mixed(args):
    """Oracle mixed round on one host core: each step is a slice of the
    mixed workload (one prefill prompt's last 8 query rows + 4 decode
    requests)."""
    import numpy as np
    import torch
    import oracle
    from paged_kv_cache_307_gb300 import workloads as W
    c = W.mixed_case(device="cpu", n_prefill=1, n_decode=4, chunk=8, nan_fill=False)
    f64 = lambda t: t.to(torch.float64).numpy()
    k, v, q = f64(c["k_cache"]), f64(c["v_cache"]), f64(c["q"])
    qs, lens, tables = c["query_start"].numpy(), c["context_lens"].numpy(), c["block_tables"].numpy()
    flops = W.varlen_flops(lens, np.diff(qs), q.shape[1], q.shape[2])
    for _ in range(args.warmup):
        oracle.paged_prefill_varlen(q, qs, k, v, tables, lens, c["scale"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.paged_prefill_varlen(q, qs, k, v, tables, lens, c["scale"])
    dt = time.perf_counter() - t0
    val = flops * args.steps / dt / 1e12
    line = {"impl": "reference", "metric": "mixed round attention TFLOP/s (bf16, unmasked work)",
            "value": round(val, 6), "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "mixed: " + WORKLOAD_TEXT["mixed"],
                       "sample": "one 8-row prefill slice + 4 decode requests per step"},
            "cpu_baseline": {"value": round(val, 6), "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
                             "sample": "%d steps of one 8-row prefill slice + 4 decode requests" % args.steps},
            "e2e": {"value": round(val, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle timed on one host core: each step is one (sequence, KV head)
    slice of the workload (append + decode), cycling through a 16-sequence
    sample, so K steps stay within minutes."""
    if rank != 0:
        return
    if args.workload == "c5prefill":
        return run_reference_prefill(args)
    if args.workload == "swap":
        return run_reference_swap(args)
    if args.workload == "mixed":
        return run_reference_mixed(args)
    fp8 = args.workload.endswith("fp8")
    tasks, nbytes = (_cpu_tasks_fp8 if fp8 else _cpu_tasks)(args.workload, 16, seed=12345)
    fn = _oracle_seq_fp8 if fp8 else _oracle_slice
    for i in range(args.warmup):
        fn(tasks[i % len(tasks)])
    t0 = time.perf_counter()
    done = 0.0
    for i in range(args.steps):
        fn(tasks[i % len(tasks)])
        done += nbytes[i % len(tasks)]
    dt = time.perf_counter() - t0
    step = dt / args.steps
    gbs = done / dt / 1e9
    unit = "sequence" if fp8 else "(sequence, KV head) slice"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 5), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(step * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload + ": " + WORKLOAD_TEXT[args.workload],
                   "sample": "one %s per step" % unit},
        "cpu_baseline": {"value": round(gbs, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "%d %ss of a 16-sequence sample of workload %s "
                                   "(append + decode, float64, one thread)" % (args.steps, unit, args.workload)},
        "e2e": {"value": round(gbs, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg

def tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["bf16_tflops_sustained"]), "measured sustained"
    except Exception:
        return 1700.0, "fallback sustained"


def run_prefill(args, rank, world, local_rank):
    """The c5 chunked-prefill tile: pa_prefill_paged over 64 prompts x 512
    queries.  Metric: TFLOP/s of the unmasked causal work (QK^T and PV, two
    flops per multiply-add)."""
    import torch
    import torch.distributed as dist
    from paged_kv_cache_307_gb300 import build as B
    B.build()
    from paged_kv_cache_307_gb300 import _lib as pa
    from paged_kv_cache_307_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    case = W.prefill_case(device=dev, seed=W.SPECS["c5"].seed + 1000 * rank, nan_fill=False,
                          prompts=args.batch or None)
    q = case["q"]
    P, Tq, Hq, D = q.shape
    out = torch.empty_like(q)
    lens = case["context_lens"].cpu().numpy()
    flops = W.prefill_flops(lens, Tq, Hq, D)
    stream = torch.cuda.current_stream()

    def step(qq=q, tables=case["block_tables"], cl=case["context_lens"]):
        pa.prefill(out, qq, case["k_cache"], case["v_cache"], tables, cl, case["scale"])

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert pa.last_error() == 0
    K = args.steps
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    sampler = ClockSampler(int(vis[local_rank]) if len(vis) > local_rank and vis[local_rank].isdigit()
                           else local_rank)
    sampler.start()
    time.sleep(0.25)
    sampler.begin()
    start.record(stream)
    for _ in range(K):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    sampler.end()
    clocks = sampler.stop()
    total_ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    assert pa.last_error() == 0
    step_s = total_ms / 1e3 / K
    tflops = world * flops / step_s / 1e12

    # end to end: Q uploaded and the output read back every step, overlapped
    # with the neighbouring steps' compute
    Ke = min(K, 100)
    e2e_ms, _, h2d, d2h = pipelined_e2e(
        stream, {"q": q.cpu().pin_memory()}, out,
        lambda d, o: pa.prefill(o, d["q"], case["k_cache"], case["v_cache"], case["block_tables"],
                                case["context_lens"], case["scale"]), Ke)
    e2e_s = max_over_ranks(e2e_ms, world, dev) / 1e3 / Ke
    if rank != 0:
        return
    peak, src = tensor_peak()
    line = {
        "metric": "chunked-prefill tile TFLOP/s (bf16, causal, unmasked work)", "value": round(tflops, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(total_ms / K, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "c5prefill: " + WORKLOAD_TEXT["c5prefill"], "prompts": P, "queries": Tq,
                   "num_heads": Hq, "num_kv_heads": case["k_cache"].shape[2], "head_dim": D,
                   "flops_per_step": flops,
                   "l2": "K/V %.2f GB + Q/O %.2f GB per call (larger than L2); no flush"
                         % (2 * case["k_cache"].numel() * 2 / 1e9, 2 * q.numel() * 2 / 1e9)},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tflops / peak, 4), "traffic": None,
                     "kernel": "prefill_kernel (tcgen05.mma, TMEM accumulators)",
                     "peak_source": "%s bf16 (MEASURED_PEAKS.json)" % src},
        "e2e": {"value": round(world * flops / e2e_s / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "Q uploaded and output read back every step, double-buffered on a copy stream"},
        "gpu_launches": K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_swap(args, rank, world, local_rank):
    """Swap-out then swap-in of 4096 blocks (pa_swap_blocks both ways).
    Metric: GB/s of K/V bytes moved over the host link (both directions).
    The copy engine moving the same bytes as one contiguous transfer each
    way is timed beside it as the link's measured rate."""
    import numpy as np
    import torch
    from paged_kv_cache_307_gb300 import build as B
    B.build()
    from paged_kv_cache_307_gb300 import _lib as pa

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    NB, bs, H, D, n = 8192, 16, 32, 128, args.batch or 4096
    g = torch.Generator(device=dev).manual_seed(4242 + rank)
    k = torch.randn(NB, bs, H, D, device=dev, generator=g).to(torch.bfloat16)
    v = torch.randn(NB, bs, H, D, device=dev, generator=g).to(torch.bfloat16)
    hk = torch.empty((n, bs, H, D), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    rng = np.random.default_rng(7 + rank)
    perm = rng.permutation(NB)
    out_pairs = torch.from_numpy(np.stack([perm[:n], np.arange(n)], 1)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(n), perm[n:2 * n] if 2 * n <= NB else perm[:n]], 1)).to(dev)
    block_bytes = bs * H * D * 2
    moved = 2 * 2 * n * block_bytes                      # K and V, out and back
    stream = torch.cuda.current_stream()

    def step():
        pa.swap_blocks(hk, hv, k, v, out_pairs)
        pa.swap_blocks(k, v, hk, hv, in_pairs)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert pa.last_error() == 0
    K = min(args.steps, 200)
    e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    sampler = ClockSampler(int(vis[local_rank]) if len(vis) > local_rank and vis[local_rank].isdigit()
                           else local_rank)
    sampler.start()
    time.sleep(0.25)
    sampler.begin()
    e[0].record(stream)
    for _ in range(K):
        step()
    e[1].record(stream)
    torch.cuda.synchronize()
    sampler.end()
    clocks = sampler.stop()
    assert pa.last_error() == 0
    ms = max_over_ranks(e[0].elapsed_time(e[1]), world, dev) / K
    value = whole_job_rate(moved, ms, 1, world) / 1e9
    # copy engine, same bytes, contiguous, both directions
    flat_d = k[:n].view(-1)
    flat_h = hk.view(-1)
    for _ in range(3):
        flat_h.copy_(flat_d, non_blocking=True)
        flat_d.copy_(flat_h, non_blocking=True)
    torch.cuda.synchronize()
    Kc = min(K, 50)
    e[0].record(stream)
    for _ in range(Kc):
        for _ in range(2):                               # K and V
            flat_h.copy_(flat_d, non_blocking=True)
            flat_d.copy_(flat_h, non_blocking=True)
    e[1].record(stream)
    torch.cuda.synchronize()
    ce_gbs = moved / (e[0].elapsed_time(e[1]) / Kc / 1e3) / 1e9
    if rank != 0:
        return
    line = {
        "metric": "KV block swap GB/s (device <-> page-locked host, both directions)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "swap: " + WORKLOAD_TEXT["swap"], "blocks": n, "block_bytes_kv": 2 * block_bytes,
                   "bytes_per_step": moved, "l2": "1.07 GB each way, larger than L2; no flush"},
        "roofline": {"bound": "host link", "achieved": round(value, 2), "peak": round(ce_gbs, 2), "unit": "GB/s",
                     "frac": round(value / ce_gbs, 4), "traffic": None,
                     "kernel": "swap_blocks_kernel (copies over NVLink-C2C from SM loads/stores)",
                     "peak_source": "copy engine moving the same bytes contiguously, measured in this run"},
        "e2e": {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": moved // 2,
                "d2h_bytes_per_step": moved // 2, "note": "the swap is itself the host transfer"},
        "gpu_launches": 2 * K,
        "clocks": clocks,
    }
    if world == 1 and not args.no_cpu_baseline:
        sample = _swap_sample(64, 5)
        t0, reps = time.perf_counter(), 0
        while time.perf_counter() - t0 < min(args.cpu_seconds, 5.0):
            swap_cpu_once(sample)
            reps += 1
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": round(reps * 2 * 2 * 64 * block_bytes / dt / 1e9, 4), "unit": "GB/s",
                                "cores": 1, "kind": "oracle",
                                "sample": "%d repetitions of 64 blocks out and back (numpy copies)" % reps}
    print(json.dumps(line), flush=True)


def run_mixed(args, rank, world, local_rank):
    """One mixed round (decode requests + prefill chunks) through
    pa_prefill_varlen.  Metric: TFLOP/s of the unmasked causal work.  The
    same round as two calls (the chunks through pa_prefill_paged, the decode
    requests through pa_decode) is timed beside it."""
    import numpy as np
    import torch
    from paged_kv_cache_307_gb300 import build as B
    B.build()
    from paged_kv_cache_307_gb300 import _lib as pa
    from paged_kv_cache_307_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    case = W.mixed_case(device=dev, seed=W.SPECS["c5"].seed + 1000 * rank, nan_fill=False)
    q = case["q"]
    rows, Hq, D = q.shape
    out = torch.empty_like(q)
    lens = case["context_lens"].cpu().numpy()
    qs = case["query_start"].cpu().numpy()
    nq = np.diff(qs)
    flops = W.varlen_flops(lens, nq, Hq, D)
    npf, ndec = case["n_prefill"], case["n_decode"]
    Hkv = case["k_cache"].shape[2]
    kv_bytes = int(lens.sum()) * 2 * Hkv * D * 2
    stream = torch.cuda.current_stream()

    def step(qq=q):
        pa.prefill_varlen(out, qq, case["query_start"], case["k_cache"], case["v_cache"], case["block_tables"],
                          case["context_lens"], case["scale"])

    # the same round as two calls
    chunk = int(nq[0]) if npf else 0
    q_pf = q[:npf * chunk].reshape(npf, chunk, Hq, D) if npf else None
    out_pf = torch.empty_like(q_pf) if npf else None
    q_dec = q[npf * chunk:].contiguous()
    out_dec = torch.empty_like(q_dec)
    tab_pf, tab_dec = case["block_tables"][:npf].contiguous(), case["block_tables"][npf:].contiguous()
    len_pf, len_dec = case["context_lens"][:npf].contiguous(), case["context_lens"][npf:].contiguous()
    ws = pa.alloc_workspace(q_dec, case["k_cache"], tab_dec)

    def split_step():
        if npf:
            pa.prefill(out_pf, q_pf, case["k_cache"], case["v_cache"], tab_pf, len_pf, case["scale"])
        pa.decode(out_dec, q_dec, case["k_cache"], case["v_cache"], tab_dec, len_dec, case["scale"], workspace=ws)

    def timed(fn, K):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(K):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K

    K = min(args.steps, 500)
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    sampler = ClockSampler(int(vis[local_rank]) if len(vis) > local_rank and vis[local_rank].isdigit()
                           else local_rank)
    sampler.start()
    time.sleep(0.25)
    sampler.begin()
    ms = max_over_ranks(timed(step, K), world, dev)
    sampler.end()
    clocks = sampler.stop()
    assert pa.last_error() == 0
    split_ms = timed(split_step, K)
    assert pa.last_error() == 0
    e2e_ms, _, h2d, d2h = pipelined_e2e(
        stream, {"q": q.cpu().pin_memory()}, out,
        lambda d, o: pa.prefill_varlen(o, d["q"], case["query_start"], case["k_cache"], case["v_cache"],
                                       case["block_tables"], case["context_lens"], case["scale"]), min(K, 100))
    e2e_ms = max_over_ranks(e2e_ms, world, dev) / min(K, 100)
    if rank != 0:
        return
    peak, src = tensor_peak()
    tflops = world * flops / (ms / 1e3) / 1e12
    line = {
        "metric": "mixed round attention TFLOP/s (bf16, unmasked work)", "value": round(tflops, 2),
        "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "mixed: " + WORKLOAD_TEXT["mixed"], "prefill_chunks": int(npf),
                   "decode_requests": int(ndec), "query_rows": int(rows), "flops_per_step": flops,
                   "kv_bytes_per_step": kv_bytes, "l2": "K/V pool larger than L2; no flush"},
        "kv_gbs": round(kv_bytes / (ms / 1e3) / 1e9, 2),
        "tokens_per_s": round(world * rows / (ms / 1e3), 1),
        "split_calls": {"ms_per_step": round(split_ms, 5),
                        "note": "the same round as pa_prefill_paged (chunks) + pa_decode (decode requests)"},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tflops / peak, 4), "traffic": None,
                     "kernel": "prefill_kernel over ragged query counts (tcgen05.mma, TMEM accumulators)",
                     "peak_source": "%s bf16 (MEASURED_PEAKS.json)" % src},
        "e2e": {"value": round(world * flops / (e2e_ms / 1e3) / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "Q uploaded and output read back every step, double-buffered on a copy stream"},
        "gpu_launches": K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch
    import torch.distributed as dist

    from paged_kv_cache_307_gb300 import build as B
    B.build()
    from paged_kv_cache_307_gb300 import _lib as pa
    from paged_kv_cache_307_gb300 import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    fp8 = args.workload.endswith("fp8")
    base = args.workload[:-3] if fp8 else args.workload
    spec = W.SPECS[base]
    case = W.decode_case(base, device=dev, nan_fill=False, seed=spec.seed + 1000 * rank, B=args.batch or None)
    if fp8:
        case = W.fp8_case(case)
        k_scale, v_scale = case.extra["k_scale"], case.extra["v_scale"]
    Bsz, Hq, D = case.q.shape
    # workloads whose samples share prompt blocks run the shared-prefix call
    shared = "group_start" in case.extra and not fp8 and not args.no_share
    if shared:
        gs, sb = case.extra["group_start"], case.extra["shared_blocks"]
        ws = pa.alloc_shared_workspace(case.q, case.k_cache, case.block_tables, sb.shape[0], args.partition)
    else:
        ws = pa.alloc_workspace(case.q, case.k_cache, case.block_tables, args.partition)
    out = torch.empty_like(case.q)
    stream = torch.cuda.current_stream()
    P = pa.partition_size(Bsz, Hq, spec.Hkv, D, case.max_blocks, spec.bs, args.partition, fp8=fp8)
    # append + decode; a split call adds the merge and, with its workspace
    # holding the work-item counter, the kernel that clears it
    launches_per_step = 4 if shared else 2 + (2 if case.max_blocks * spec.bs > P else 0)

    # HBM bytes a decode call must move: each physical block once (shared
    # prompt blocks count once; for private blocks this is the logical count)
    logical_bytes = W.algorithmic_decode_bytes(case)
    dec_bytes = W.unique_decode_bytes(case)
    app_bytes = W.append_bytes(case)
    step_bytes = dec_bytes + app_bytes

    def append(key=None, value=None, slots=None):
        key = case.key if key is None else key
        value = case.value if value is None else value
        slots = case.slot_mapping if slots is None else slots
        if fp8:
            pa.reshape_and_cache_fp8(key, value, slots, case.k_cache, case.v_cache, k_scale, v_scale)
        else:
            pa.reshape_and_cache(key, value, slots, case.k_cache, case.v_cache)

    def decode(q=None, tables=None, lens=None):
        q = case.q if q is None else q
        tables = case.block_tables if tables is None else tables
        lens = case.context_lens if lens is None else lens
        if fp8:
            pa.decode_fp8(out, q, case.k_cache, case.v_cache, k_scale, v_scale, tables, lens, case.scale,
                          partition_size=args.partition, workspace=ws)
        elif shared:
            pa.decode_shared(out, q, case.k_cache, case.v_cache, tables, lens, gs, sb, case.scale,
                             partition_size=args.partition, workspace=ws)
        else:
            pa.decode(out, q, case.k_cache, case.v_cache, tables, lens, case.scale,
                      partition_size=args.partition, workspace=ws)

    for _ in range(max(args.warmup, 3)):
        append()
        decode()
    torch.cuda.synchronize()
    assert pa.last_error() == 0, "device-detected error during warm-up"

    K = args.steps
    d0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    d1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    vis = [x for x in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if x.strip()]
    sampler = ClockSampler(int(vis[local_rank]) if len(vis) > local_rank and vis[local_rank].isdigit()
                           else local_rank)
    sampler.start()
    time.sleep(0.25)
    sampler.begin()
    start.record(stream)
    for i in range(K):
        append()
        d0[i].record(stream)
        decode()
        d1[i].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    sampler.end()
    clocks = sampler.stop()
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(stop), world, dev)
    dec_ms = statistics.mean(d0[i].elapsed_time(d1[i]) for i in range(K))
    assert pa.last_error() == 0, "device-detected error in the timed region"
    step_s = total_ms / 1e3 / K
    value = whole_job_rate(step_bytes, total_ms, K, world) / 1e9

    # a longer repeat of the same step with no per-call events, beside the
    # K-step region: a steadier step time and a fuller clock record when K is
    # small (the line's value stays the K-step one)
    repeat_line = None
    R = max(K, args.long_repeat)
    if R > K:
        ra, rb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        rs = ClockSampler(sampler.index)
        rs.start()
        time.sleep(0.25)
        rs.begin()
        ra.record(stream)
        for _ in range(R):
            append()
            decode()
        rb.record(stream)
        torch.cuda.synchronize()
        rs.end()
        r_clocks = rs.stop()
        assert pa.last_error() == 0, "device-detected error in the long repeat"
        r_ms = ra.elapsed_time(rb) / R
        repeat_line = {"steps": R, "ms_per_step": round(r_ms, 5),
                       "value": round(world * step_bytes / (r_ms / 1e3) / 1e9, 2), "unit": "GB/s",
                       "clocks": r_clocks, "note": "append + decode, no per-call events, after the K-step region"}

    # the same step captured once as a CUDA graph and replayed K times
    graph_line = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            append()
            decode()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            append()
            decode()
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        ga, gb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ga.record(stream)
        for _ in range(K):
            graph.replay()
        gb.record(stream)
        torch.cuda.synchronize()
        assert pa.last_error() == 0, "device-detected error in graph replay"
        g_ms = ga.elapsed_time(gb) / K
        graph_line = {"ms_per_step": round(g_ms, 5), "value": round(world * step_bytes / (g_ms / 1e3) / 1e9, 2),
                      "unit": "GB/s", "steps": K, "note": "append + decode captured once, replayed per step"}
        del graph
    except RuntimeError as exc:
        graph_line = {"error": str(exc).splitlines()[0][:200]}

    # end to end through the public API (inputs uploaded and the result read
    # back every step, overlapped with the neighbouring steps' compute)
    host = {n: getattr(case, n).cpu().pin_memory() for n in ("q", "key", "value", "slot_mapping",
                                                             "block_tables", "context_lens")}
    if shared:
        host["group_start"], host["shared_blocks"] = gs.cpu().pin_memory(), sb.cpu().pin_memory()

    def e2e_compute(d, o):
        if fp8:
            pa.reshape_and_cache_fp8(d["key"], d["value"], d["slot_mapping"], case.k_cache, case.v_cache,
                                     k_scale, v_scale)
            pa.decode_fp8(o, d["q"], case.k_cache, case.v_cache, k_scale, v_scale, d["block_tables"],
                          d["context_lens"], case.scale, partition_size=args.partition, workspace=ws)
        elif shared:
            pa.reshape_and_cache(d["key"], d["value"], d["slot_mapping"], case.k_cache, case.v_cache)
            pa.decode_shared(o, d["q"], case.k_cache, case.v_cache, d["block_tables"], d["context_lens"],
                             d["group_start"], d["shared_blocks"], case.scale, partition_size=args.partition,
                             workspace=ws)
        else:
            pa.reshape_and_cache(d["key"], d["value"], d["slot_mapping"], case.k_cache, case.v_cache)
            pa.decode(o, d["q"], case.k_cache, case.v_cache, d["block_tables"], d["context_lens"], case.scale,
                      partition_size=args.partition, workspace=ws)

    if world > 1:
        dist.barrier()
    Ke = min(K, 1000)
    e2e_ms, e2e_last, h2d, d2h = pipelined_e2e(stream, host, out, e2e_compute, Ke)
    e2e_ms = max_over_ranks(e2e_ms, world, dev)
    e2e_value = whole_job_rate(step_bytes, e2e_ms, Ke, world) / 1e9
    # the pipelined results equal the device-resident step's
    assert torch.equal(e2e_last, out.cpu()), "end-to-end result differs from the device-resident step"

    if rank != 0:
        return
    peak, peak_src = peaks()
    achieved = dec_bytes / (dec_ms / 1e3) / 1e9
    traffic = traffic_record(args.workload, Bsz, SHARED_SOURCES if shared else FP8_SOURCES if fp8 else DECODE_SOURCES)
    kname = ("pa_decode_shared (shared_decode_kernel + shared_merge_kernel)" if shared else
             "pa_decode_fp8 (decode_kernel + merge_kernel)" if fp8 else "pa_decode (decode_kernel + merge_kernel)")
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 K/V, bf16 Q/O, f32 math" if fp8 else ("bf16" if spec.dtype == "bf16" else "f32"),
        "data": "synthetic",
        "config": {"workload": args.workload + ": " + WORKLOAD_TEXT[args.workload], "batch": Bsz,
                   "num_heads": Hq, "num_kv_heads": spec.Hkv, "head_dim": D, "block_size": spec.bs,
                   "partition_tokens": P, "pool_bytes": 2 * case.k_cache.numel() * case.k_cache.element_size(),
                   "kv_dtype": "e4m3 + per-token fp32 scales" if fp8 else spec.dtype,
                   "l2": "inputs larger than L2 (K/V pool %.2f GB vs 129 MB L2); no flush"
                         % (2 * case.k_cache.numel() * case.k_cache.element_size() / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "step_bytes": step_bytes, "decode_bytes": dec_bytes, "append_bytes": app_bytes,
                   "decode_logical_bytes": logical_bytes,
                   "shared_prefix": bool(shared)},
        "seq_steps_per_s": round(world * Bsz / step_s, 1),
        "pct_of_peak": round(100.0 * value / peak, 2),
        "logical_gbs": round(logical_bytes / (dec_ms / 1e3) / 1e9, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "bytes_per_launch": dec_bytes,
                     "traffic_over_bytes": round(traffic / dec_bytes, 4) if traffic else None,
                     "kernel": "%s, %.4f ms per call" % (kname, dec_ms),
                     "peak_source": "%s (MEASURED_PEAKS.json hbm_gbs)" % peak_src if peak_src == "measured"
                     else "fallback 6.8 TB/s"},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke, "ms_per_step": round(e2e_ms / Ke, 5),
                "note": "inputs uploaded and result read back every step, double-buffered on a copy stream"},
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
        "graph": graph_line,
        "long_repeat": repeat_line,
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[v] = "1"
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        if args.workload == "c5prefill":
            run_prefill(args, rank, world, local_rank)
        elif args.workload == "swap":
            run_swap(args, rank, world, local_rank)
        elif args.workload == "mixed":
            run_mixed(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python3
"""Benchmark of the paged-attention hot path on one GB300 (or N independent replicas).

One step = one serving step of the path: ``pa_reshape_and_cache`` writes this step's new K/V
tokens into the paged pool, then ``pa_attention`` runs the block-table-indirected attention
(decode partitions, chunked-prefill tiles when the batch has them, and the log-sum-exp merge).
The default workload is the 32 x 8k Llama-3-70B-shaped decode step (one layer): 32 sequences
of 8192 keys, 64 query / 8 KV heads, head_dim 128, block size 16, blocks randomly placed.

Prints ONE JSON line.  ``value`` is the effective KV bandwidth: algorithmic bytes of the step
(K/V of every attended token of every sequence, Q, output, used block-table entries and the
batch descriptor, plus the new tokens read and written by the scatter) / device time of the
step.  L2 is flushed (a 512 MiB write) before every timed step, outside the timed events.

``--impl reference`` times the fp64 CPU oracle on this machine's host cores instead (a bounded
sample of the same workload per step); there is no GPU reference implementation.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-attention KV GB/s and % of HBM roofline; decode tok/s per layer"
DEFAULT_WORKLOAD = "llama70b_32x8k_decode"
FLUSH_BYTES = 512 << 20


# ------------------------------------------------------------------------------ bookkeeping

def shared_prefix_tokens(b) -> int:
    """Keys of the prefix every sequence shares, rounded down to whole 512-key partitions, when
    the batch qualifies for the shared-prefix pass (decode rows only); else 0."""
    sp = (int(b.meta.get("shared_prefix_len", 0)) // 512) * 512
    ok = b.max_query_len == 1 and sp < b.max_seq_len
    return sp if ok else 0


def shared_prefix_kernel(b, sp: int, num_sms: int = 152) -> str:
    """The kernel pa_attention picks for the shared-prefix pass: one Q tile per CTA while the
    two-tile grid (2 x 128 // G rows per CTA, every kv head and prefix partition) would not
    fill the GPU's SMs."""
    rows_pair = 2 * (128 // (b.num_q_heads // b.num_kv_heads))
    ctas = -(-b.num_tokens // rows_pair) * b.num_kv_heads * (sp // 512)
    return "prefill_parity_kernel" if ctas < num_sms else "prefill_pair_kernel"


def algorithmic_bytes(b, sp: int = 0) -> dict:
    """Bytes the step must move at minimum.  K/V are counted per attended token of every
    sequence ("logical"); "unique" counts each physical (block, offset) slot once, which is what
    the roofline of an aliased-prefix batch is measured against.  With a shared-prefix pass over
    the first ``sp`` keys, the decode kernel's share is the keys past them and the pass's share
    the prefix's K/V once plus every row's query."""
    hkv, d, bs = b.num_kv_heads, b.head_dim, b.block_size
    eb = 1 if b.kv_dtype == "e4m3" else 2  # bytes per cached value (E4M3 or fp16)
    row_kv = hkv * d * eb * 2  # K and V of one token, all kv heads
    lens = np.array([s.seq_len for s in b.seqs], dtype=np.int64)
    qlens = np.array([s.query_len for s in b.seqs], dtype=np.int64)
    active = qlens > 0
    kv_logical = int(lens[active].sum()) * row_kv
    slots = []
    bt = b.block_tables.numpy().astype(np.int64)
    for s in np.nonzero(active)[0]:
        pos = np.arange(lens[s])
        slots.append(bt[s, pos // bs] * bs + pos % bs)
    kv_unique = (np.unique(np.concatenate(slots)).size if slots else 0) * row_kv
    t = b.num_tokens
    q_bytes = t * b.num_q_heads * d * 2
    out_bytes = q_bytes
    table = int(((lens[active] + bs - 1) // bs).sum()) * 4
    desc = b.num_seqs * 4 + (b.num_seqs + 1) * 4
    t_new = int(b.k_new.shape[0])
    cache = t_new * hkv * d * 2 * (2 + eb) + t_new * 8  # fp16 K/V read, cache values written
    attn = q_bytes + out_bytes + table + desc

    def flops(sel):
        return int(sum(4 * b.num_q_heads * d * (s.seq_len * s.query_len -
                                                 s.query_len * (s.query_len - 1) // 2)
                       for s, keep in zip(b.seqs, sel) if keep))

    def kernel_bytes(sel, first=0):
        """Unique K/V slots (positions >= first) of the selected sequences, their Q/out rows and
        table entries."""
        idx = np.nonzero(sel)[0]
        if idx.size == 0:
            return 0
        uniq = np.unique(np.concatenate([slots[int(np.nonzero(np.nonzero(active)[0] == s)[0][0])][first:]
                                         for s in idx])).size * row_kv
        rows = int(qlens[idx].sum())
        return (uniq + 2 * rows * b.num_q_heads * d * 2 +
                int(((lens[idx] + bs - 1) // bs).sum()) * 4 + desc)

    # the decode kernel serves one-row sequences, and every sequence on the verify path
    dec = (qlens >= 1) if verify_path(b) else (qlens == 1)
    pre = (qlens > 1) & ~dec
    return {
        "kv_logical": kv_logical, "kv_unique": kv_unique,
        "attention_logical": kv_logical + attn, "attention_unique": kv_unique + attn,
        "reshape_and_cache": cache,
        "step_logical": kv_logical + attn + cache,
        "decode_rows": int((qlens == 1).sum()),
        "flops": flops(active),
        # what each attention kernel must move / compute: the decode-partition kernel serves the
        # one-row sequences, the chunked-prefill kernel the sequences with several rows
        "decode_kernel_bytes": kernel_bytes(dec, sp),
        "prefill_kernel_bytes": kernel_bytes(pre),
        "prefill_kernel_flops": flops(pre),
        "prefill_kernel": ("prefill_parity_kernel" if b.max_query_len <= 128 // (b.num_q_heads //
                                                                               hkv)
                           else "prefill_pair_kernel"),
        "shared_prefix_tokens": sp,
        "shared_prefix_kernel_bytes": sp * row_kv + q_bytes if sp else 0,
        "shared_prefix_kernel_flops": 4 * b.num_q_heads * d * sp * t if sp else 0,
    }


def verify_path(b) -> bool:
    """pa_attention serves every row with the decode kernel when each sequence has at most a
    few query rows: max_query_len x G <= 8 columns, or <= 32 over an FP8 cache."""
    cols = b.max_query_len * (b.num_q_heads // b.num_kv_heads)
    return b.max_query_len > 1 and (cols <= 8 or (b.kv_dtype == "e4m3" and cols <= 32))


def all_prefill(b) -> bool:
    """Every sequence has several query rows and the prefill kernel serves them: pa_attention
    then makes no decode launches."""
    return not verify_path(b) and b.max_query_len > 1 and b.num_prefill_seqs == b.num_seqs


def prefill_slice_ctas(b, num_sms: int = 152) -> int:
    """CTAs per launch of the two-tile prefill kernel beside decode rows, as pa_attention chooses
    them (0: one full grid): two thirds of the SMs when the decode rows' estimated SM time is at
    least 0.8 of the prefill rows' ((decode rows / prefill rows) / G x 70, halved over FP8)."""
    group = b.num_q_heads // b.num_kv_heads
    decode_rows = b.num_seqs - b.num_prefill_seqs
    prefill_rows = max(b.num_tokens - decode_rows, 1)
    r = decode_rows / prefill_rows / group * 70.0 * (0.5 if b.kv_dtype == "e4m3" else 1.0)
    return num_sms * 2 // 3 if r >= 0.8 else 0


def prefill_launches(b, decode: bool, num_sms: int = 152) -> int:
    """Launches of the chunked-prefill kernel in one call: one, except for the two-tile kernel
    beside decode rows, which may go as launches of prefill_slice_ctas CTAs each over its items
    (pairs of 128-row Q tiles x kv heads x prefill sequences)."""
    if b.max_query_len <= 1 or verify_path(b):
        return 0
    group = b.num_q_heads // b.num_kv_heads
    if b.max_query_len <= 128 // group or not decode:
        return 1
    per = prefill_slice_ctas(b, num_sms)
    if per == 0:
        return 1
    items = -(-b.max_query_len // (2 * (128 // group))) * b.num_kv_heads * b.num_prefill_seqs
    return -(-items // per)


def launches_per_step(b, sp: int = 0, num_sms: int = 152) -> int:
    parts = max(1, math.ceil(b.max_seq_len / 512))
    decode = not all_prefill(b)
    n = 1 if b.k_new.shape[0] > 0 else 0        # reshape_and_cache
    n += 1 if decode else 0                       # decode partitions
    n += prefill_launches(b, decode, num_sms)     # chunked-prefill tiles
    n += 1 if parts > 1 and decode else 0         # log-sum-exp merge
    n += 1 if sp else 0                           # shared-prefix pass
    return n


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, world: int) -> float:
    """Max of a per-rank scalar over all ranks (identity when world == 1)."""
    if world == 1:
        return x
    import torch.distributed as dist
    backend = dist.get_backend()
    dev = torch.device("cuda", torch.cuda.current_device()) if backend == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def load_peaks() -> dict:
    """HBM and dense fp16 tensor peaks: the measured ones when MEASURED_PEAKS.json is present
    (a STREAM-style copy; a cuBLAS bf16 GEMM burst, and fp16 has bf16's nominal rate), else the
    fallback figures of one earlier GB300 measurement."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return {"hbm_gbs": float(p["hbm_gbs"]),
                "hbm_src": "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)",
                "tflops": float(p["bf16_tflops"]),
                "tflops_src": "measured (MEASURED_PEAKS.json bf16_tflops burst; fp16 = bf16 "
                              "nominal rate)"}
    return {"hbm_gbs": 6800.0, "hbm_src": "fallback (6.8 TB/s, one earlier GB300 measurement)",
            "tflops": 1900.0, "tflops_src": "fallback (1.9 PFLOP/s bf16 burst, one earlier GB300 "
                                            "measurement; fp16 = bf16 nominal rate)"}


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str, interval_ms: int = 20):
        self.uuid = uuid
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.interval_ms)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.6)  # let nvidia-smi start sampling before the timed region

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def mark_load(self, t0: float, t1: float):
        """The host-clock window of a stretch of back-to-back GPU work (the clock soak)."""
        self.load = (t0, t1)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, power, reasons, load_sm, load_power = [], [], [], set(), [], []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = getattr(self, "load", (None, None))
        for t, line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            u = f[0]
            if self.uuid and self.uuid not in u and u not in self.uuid:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            # a sample read in the soak window, past its first 100 ms, was taken under load
            if lo is not None and lo + 0.1 <= t <= hi:
                load_sm.append(sm[-1])
                load_power.append(power[-1])
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        res = {"sm_mhz": statistics.median(load_sm or sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None,
               "power_w_max": max(power) if power else None,
               "samples": len(sm), "samples_under_load": len(load_sm),
               "sm_mhz_under_load_median": statistics.median(load_sm) if load_sm else None,
               "power_w_under_load_median": statistics.median(load_power) if load_power else None,
               "reasons": sorted(reasons)}
        return res


# ------------------------------------------------------------------------------ our arm

def workload_config(name, b, sp, world) -> dict:
    """The ``config`` object of a line (both arms echo the same keys)."""
    return {"workload": name, "num_seqs": b.num_seqs, "max_seq_len": b.max_seq_len,
            "max_query_len": b.max_query_len, "num_tokens": b.num_tokens,
            "num_q_heads": b.num_q_heads, "num_kv_heads": b.num_kv_heads,
            "head_dim": b.head_dim, "block_size": b.block_size, "num_blocks": b.num_blocks,
            "kv_cache_dtype": b.kv_dtype, "partition_tokens": 512,
            "shared_prefix_tokens": sp,
            "parallelism": f"replicas x{world}",
            "l2": "flushed before every timed step (512 MiB write, outside the events)"}


# The other workloads of the task's configurations, measured beside the default line: the tiny
# GQA decode, the Llama-3-8B decode, the prefix-shared decode and the mixed continuous-batching
# step over 16- and 32-token blocks.
EXTRA_WORKLOADS = ("tiny_decode", "llama8b_decode", "prefix_shared_decode", "mixed_step_bs16",
                   "mixed_step_bs32")


def measure(name, args, world, rank, dev, soak_s=0.0, clocks=None, cpu_seconds=None) -> dict:
    """One workload: K timed steps (device-resident inputs), K steps with per-kernel events,
    optionally a clock soak, the end-to-end pass from pinned host buffers and the oracle's CPU
    baseline.  Returns the workload's line (without ``clocks``)."""
    import paged_kv_cache_290_gb300 as pa
    from paged_kv_cache_290_gb300 import workloads as W

    b = W.WORKLOADS[name](keep_contiguous=False, keep_pre=False)
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sp = 0 if args.no_shared_prefix else shared_prefix_tokens(b)
    nbytes = algorithmic_bytes(b, sp)
    if sp:
        nbytes["shared_prefix_kernel"] = shared_prefix_kernel(b, sp, num_sms)
    stream = torch.cuda.current_stream()

    # device-resident inputs (the pool already holds every token; the scatter rewrites the new
    # tokens' slots with the same values, exactly as a serving step would write them)
    q = b.q.to(dev)
    k_new, v_new, slots = b.k_new.to(dev), b.v_new.to(dev), b.slot_mapping.to(dev)
    kc, vc = b.k_cache.to(dev), b.v_cache.to(dev)
    bt, sl, qsl = b.block_tables.to(dev), b.seq_lens.to(dev), b.query_start_loc.to(dev)
    out = torch.empty_like(q)
    ws = torch.empty(max(1, pa.workspace_size(b.num_tokens, b.num_q_heads, b.head_dim,
                                              b.max_seq_len)), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    sc = dict(k_scale=b.k_scale, v_scale=b.v_scale) if b.kv_dtype == "e4m3" else {}

    def step(q_, k_, v_, s_, bt_, sl_, qsl_, out_):
        pa.reshape_and_cache(k_, v_, kc, vc, s_, **sc)
        pa.attention(q_, kc, vc, bt_, sl_, qsl_, b.scale, out_, b.max_query_len, b.max_seq_len,
                     workspace=ws, num_prefill_seqs=b.num_prefill_seqs,
                     shared_prefix_tokens=sp, **sc)

    for i in range(args.warmup):
        flush.fill_(i & 255)
        step(q, k_new, v_new, slots, bt, sl, qsl, out)
    torch.cuda.synchronize()
    st, bits = pa.get_device_error()
    if st != 0:
        raise RuntimeError(f"{name}: device error after warm-up: status {st} bits {bits}")

    # -------- device-resident timed region: exactly K steps, nothing between the step events
    # but the step itself
    timed = (([] if all_prefill(b) else ["decode"])
             + (["prefill"] if b.max_query_len > 1 and not verify_path(b) else [])
             + (["shared_prefix"] if sp else []))
    mk = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(mk(), mk()) for _ in range(args.steps)]
    kev = [{k: (mk(), mk()) for k in timed} for _ in range(args.steps)]
    for e in ev + [p for d_ in kev for p in d_.values()]:
        e[0].record(stream)   # torch creates an event on its first record(); the library then
        e[1].record(stream)   # re-records the kernel events around the kernels it launches
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 255)
        ev[i][0].record(stream)
        step(q, k_new, v_new, slots, bt, sl, qsl, out)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    step_ms = [a.elapsed_time(c) for a, c in ev]

    # -------- per-kernel times: K more steps with CUDA events recorded around each attention
    # kernel on the launching stream (pa_set_timing_events).  An event between two launches
    # stops the second from starting while the first drains (programmatic dependent launch),
    # so these steps run a little longer and only their kernel intervals are used.
    inst_ms = []
    for i in range(args.steps):
        flush.fill_(i & 255)
        for k, (k0, k1) in kev[i].items():
            pa.set_timing_events(k0, k1, kernel=k)
        a0, a1 = mk(), mk()
        a0.record(stream)
        step(q, k_new, v_new, slots, bt, sl, qsl, out)
        a1.record(stream)
        inst_ms.append((a0, a1))
    torch.cuda.synchronize()
    for k in timed:
        pa.set_timing_events(None, None, kernel=k)
    kern_ms = {k: statistics.mean(d_[k][0].elapsed_time(d_[k][1]) for d_ in kev) for k in timed}
    inst_step_ms = statistics.mean(a.elapsed_time(c) for a, c in inst_ms)

    # -------- clock soak: identical steps back to back (no flush) for soak_s seconds, outside
    # the reported timing, so the clock sampler sees the SMs under this workload's load
    soak = None
    if soak_s > 0 and clocks is not None:
        s0, s1 = mk(), mk()
        n_soak = 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        s0.record(stream)
        while time.perf_counter() - t0 < soak_s:
            for _ in range(16):
                step(q, k_new, v_new, slots, bt, sl, qsl, out)
            n_soak += 16
        s1.record(stream)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        clocks.mark_load(t0, t1)
        soak = {"steps": n_soak, "seconds": t1 - t0,
                "ms_per_step": s0.elapsed_time(s1) / n_soak,
                "note": "back-to-back steps without L2 flush, outside the reported timing"}
    st, bits = pa.get_device_error()
    if st != 0:
        raise RuntimeError(f"{name}: device error in timed region: status {st} bits {bits}")
    ms = statistics.mean(step_ms)
    ms_max = reduce_max(ms, world)

    # -------- end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        # the step's inputs packed in one pinned host buffer, 256-byte aligned each, so a step
        # is one host-to-device copy, the two calls, and one device-to-host copy of the output
        parts = [b.q, b.k_new, b.v_new, b.slot_mapping, b.block_tables, b.seq_lens,
                 b.query_start_loc]
        offs, tot = [], 0
        for x in parts:
            offs.append(tot)
            tot += (x.numel() * x.element_size() + 255) // 256 * 256
        hbuf = torch.empty(tot, dtype=torch.uint8).pin_memory()
        for x, o in zip(parts, offs):
            hbuf[o:o + x.numel() * x.element_size()].copy_(x.contiguous().view(-1).view(torch.uint8))
        dbuf = torch.empty(tot, dtype=torch.uint8, device=dev)
        dq, dk, dv, ds, dbt, dsl, dqsl = (
            dbuf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape)
            for x, o in zip(parts, offs))
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = tot
        d2h = hout.numel() * hout.element_size()
        n_e2e = max(3, min(args.steps, 100))
        eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_e2e)]
        for i in range(n_e2e + 2):
            flush.fill_(i & 255)
            if i >= 2:
                eev[i - 2][0].record(stream)
            dbuf.copy_(hbuf, non_blocking=True)
            step(dq, dk, dv, ds, dbt, dsl, dqsl, out)
            hout.copy_(out, non_blocking=True)
            if i >= 2:
                eev[i - 2][1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = reduce_max(statistics.mean(a.elapsed_time(c) for a, c in eev), world)
        assert torch.equal(hout.view(torch.int16), out.cpu().view(torch.int16))
        e2e = {"value": world * nbytes["step_logical"] / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": n_e2e}

    peaks = load_peaks()
    peak = peaks["hbm_gbs"]
    kernels = kernel_rooflines(nbytes, kern_ms, peaks)
    for k in kernels:
        kernels[k]["traffic"] = load_traffic(name, k)
    dominant = dominant_kernel(kernels)
    value = world * nbytes["step_logical"] / (ms_max * 1e-3) / 1e9
    tok_s = world * nbytes["decode_rows"] / (ms_max * 1e-3)
    result = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if b.kv_dtype == "bf16" else "f16",  # E4M3 codes run fp16 MMAs
        "data": "synthetic",
        "config": workload_config(name, b, sp, world),
        "decode_tok_s_per_layer": tok_s,
        "hbm_roofline_frac_step": (nbytes["step_logical"] / (ms * 1e-3) / 1e9) / peak,
        "bytes": nbytes,
        "roofline": kernels[dominant],
        "roofline_kernels": kernels,
        "gpu_launches": launches_per_step(b, sp, num_sms) * args.steps,
        "wall_ms_per_step": wall * 1e3 / args.steps,
        "kernel_timing": {"steps": args.steps, "ms_per_step_with_kernel_events": inst_step_ms,
                          "note": "per-kernel CUDA events are taken on K further steps; "
                                  "value and ms_per_step come from K steps without them"},
        "impl": "ours",
    }
    if nbytes["kv_unique"] != nbytes["kv_logical"]:
        # aliased prefix blocks: the unique bytes are what the HBM roofline divides
        result["value_unique"] = world * (nbytes["attention_unique"] +
                                          nbytes["reshape_and_cache"]) / (ms_max * 1e-3) / 1e9
        result["hbm_roofline_frac_step_unique"] = result["value_unique"] / world / peak
    if soak is not None:
        result["clock_soak"] = soak
    if e2e is not None:
        result["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(
            b, nbytes, budget_s=args.cpu_seconds if cpu_seconds is None else cpu_seconds)
    return result


def summary(res: dict) -> dict:
    """The fields of a workload's line kept in the ``workloads`` object of the default line."""
    keep = ("value", "unit", "ms_per_step", "value_unique", "decode_tok_s_per_layer",
            "hbm_roofline_frac_step", "hbm_roofline_frac_step_unique", "roofline",
            "roofline_kernels", "gpu_launches", "e2e", "cpu_baseline", "config", "dtype",
            "steps", "warmup")
    return {k: res[k] for k in keep if k in res}


def run_ours(args, world, rank, local):
    import paged_kv_cache_290_gb300 as pa
    from paged_kv_cache_290_gb300 import build as pa_build

    if rank == 0 or not os.path.exists(pa_build.LIB):
        pa_build.build()
    barrier(world)
    pa.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", ""))
    clocks = ClockSampler(uuid)
    clocks.start()
    result = measure(args.workload, args, world, rank, dev, soak_s=args.soak_seconds,
                     clocks=clocks)
    result["clocks"] = clocks.stop()
    if "clock_soak" in result and "decode" in result["roofline_kernels"]:
        mhz = result["clocks"]["sm_mhz_under_load_median"]
        if mhz:  # the decode kernel's time in SM clock cycles at the median clock under load
            result["clock_soak"]["decode_kcycles_at_median_mhz"] = (
                result["roofline_kernels"]["decode"]["ms_per_launch"] * 1e-3 * mhz * 1e3)
    if args.workload == DEFAULT_WORKLOAD and not args.no_workloads:
        extra = {}
        for name in EXTRA_WORKLOADS:
            torch.cuda.empty_cache()
            c2 = ClockSampler(uuid)
            c2.start()
            r = measure(name, args, world, rank, dev,
                        cpu_seconds=min(args.cpu_seconds, args.extra_cpu_seconds))
            r["clocks"] = c2.stop()
            extra[name] = summary(r)
            extra[name]["clocks"] = r["clocks"]
        result["workloads"] = extra
    return result


# The GB300's nominal figures, reported beside the measured ones: HBM3e ~8 TB/s and dense
# fp16/bf16 tensor throughput 2.25 PFLOP/s.
NOMINAL_HBM_GBS = 8000.0
NOMINAL_TFLOPS = 2250.0


def dominant_kernel(kernels: dict) -> str:
    """The kernel the step's `roofline` reports: the one whose own work takes longest at its roof
    (bytes / copy bandwidth or flops / tensor throughput).  Kernels that run side by side have
    overlapping event intervals, so their launch times do not say which one bounds the step."""
    return max(kernels, key=lambda k: kernels[k]["bytes_per_launch"] / kernels[k]["peak"]
               if kernels[k]["unit"] == "GB/s"
               else kernels[k]["flops_per_launch"] / (kernels[k]["peak"] * 1e3))


def kernel_rooflines(nbytes, kern_ms, peaks) -> dict:
    """Roofline of each timed attention kernel from its algorithmic bytes / flops and its mean
    live launch time.  The bound is whichever roof the kernel's arithmetic intensity hits first
    (HBM copy bandwidth vs fp16 dense tensor throughput, both measured); the fraction of the
    nominal figure of the same roof is reported too."""
    out = {}
    specs = {"decode": ("decode_partition_kernel", nbytes["decode_kernel_bytes"], 0),
             "prefill": (nbytes.get("prefill_kernel", "prefill"), nbytes["prefill_kernel_bytes"],
                         nbytes["prefill_kernel_flops"]),
             "shared_prefix": (nbytes.get("shared_prefix_kernel", "prefill kernel") +
                               " (shared-prefix pass)",
                               nbytes.get("shared_prefix_kernel_bytes", 0),
                               nbytes.get("shared_prefix_kernel_flops", 0))}
    for k, ms in kern_ms.items():
        name, nb, fl = specs[k]
        t = ms * 1e-3
        tensor = fl / (peaks["tflops"] * 1e12) > nb / (peaks["hbm_gbs"] * 1e9)
        if tensor:
            achieved, peak, unit, src = fl / t / 1e12, peaks["tflops"], "TFLOP/s", peaks["tflops_src"]
        else:
            achieved, peak, unit, src = nb / t / 1e9, peaks["hbm_gbs"], "GB/s", peaks["hbm_src"]
        nominal = NOMINAL_TFLOPS if tensor else NOMINAL_HBM_GBS
        out[k] = {"kernel": name, "bound": "tensor" if tensor else "hbm", "achieved": achieved,
                  "peak": peak, "unit": unit, "frac": achieved / peak, "peak_source": src,
                  "nominal_peak": nominal, "frac_of_nominal": achieved / nominal,
                  "traffic": None, "ms_per_launch": ms, "bytes_per_launch": nb,
                  "flops_per_launch": fl}
    return out


def load_traffic(workload, kernel="decode"):
    """DRAM bytes per launch of one kernel ("decode" or "prefill") on one workload, from the
    committed ncu summaries (profiles/traffic.json), and only while that kernel's source file
    is the one the counters were taken on (else None)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    entry = json.load(open(path)).get(workload if kernel == "decode" else f"{workload}:{kernel}")
    if not entry:
        return None
    src = os.path.join(ROOT, "paged_kv_cache_290_gb300", "csrc", entry.get("source", "pa_decode.cu"))
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return entry["dram_bytes_per_launch"] if digest == entry.get("source_sha256_16") else None


# ------------------------------------------------------------------------------ CPU oracle

def _sub_batch(b, seqs):
    """The same pool restricted to some sequences (for bounded oracle samples)."""
    idx = torch.tensor(seqs, dtype=torch.int64)
    qlens = torch.tensor([b.seqs[i].query_len for i in seqs], dtype=torch.int64)
    qsl = torch.zeros(len(seqs) + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(qlens, 0).to(torch.int32)
    rows = torch.cat([torch.arange(int(b.query_start_loc[i]), int(b.query_start_loc[i + 1]))
                      for i in seqs])
    return (b.q[rows], b.block_tables[idx], b.seq_lens[idx], qsl, rows)


def _oracle_sample_seconds(b, seqs):
    import oracle
    q, bt, sl, qsl, rows = _sub_batch(b, seqs)
    t0 = time.perf_counter()
    if b.kv_dtype == "e4m3":
        oracle.attention_fp8(q, b.k_cache, b.v_cache, bt, sl, qsl, b.scale, b.k_scale, b.v_scale)
    else:
        oracle.attention(q, b.k_cache, b.v_cache, bt, sl, qsl, b.scale)
    return time.perf_counter() - t0


def _sample_bytes(b, seqs):
    hkv, d, bs = b.num_kv_heads, b.head_dim, b.block_size
    eb = 1 if b.kv_dtype == "e4m3" else 2
    tot = 0
    for i in seqs:
        s = b.seqs[i]
        tot += s.seq_len * hkv * d * eb * 2 + 2 * s.query_len * b.num_q_heads * d * 2
        tot += ((s.seq_len + bs - 1) // bs) * 4 + 8
    return tot


def cpu_baseline(b, nbytes, budget_s=12.0):
    """The fp64 oracle, as it stands, on this host's cores: a bounded, seeded sample of the
    workload's sequences, timed 3 times (median); value in the benchmark's unit (GB/s)."""
    import oracle
    oracle.build()
    threads = oracle.get_threads()
    g = torch.Generator().manual_seed(7)
    order = torch.randperm(b.num_seqs, generator=g).tolist()
    order = [i for i in order if b.seqs[i].query_len > 0]
    probe = order[:1]
    t1 = _oracle_sample_seconds(b, probe)
    per = t1 / max(1, len(probe))
    n = max(1, min(len(order), int((budget_s / 3) / max(per, 1e-6))))
    seqs = order[:n]
    times = [_oracle_sample_seconds(b, seqs) for _ in range(3)]
    t = statistics.median(times)
    sb = _sample_bytes(b, seqs)
    res = {"value": sb / t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
           "sample": f"attention of {len(seqs)} of {b.num_seqs} sequences (all their query rows "
                     f"and heads; the scatter-write's copy is left out), fp64 C oracle with "
                     f"OpenMP, median of 3 runs of {t:.2f} s",
           "seconds": t}
    if t * threads < budget_s / 3:
        # a small sample (the tiny workload): its single-core time too
        oracle.set_threads(1)
        try:
            t1 = statistics.median(_oracle_sample_seconds(b, seqs) for _ in range(3))
        finally:
            oracle.set_threads(threads)
        res["single_core"] = {"value": sb / t1 / 1e9, "unit": "GB/s", "cores": 1, "seconds": t1}
    return res


def run_reference(args, world, rank):
    """The oracle timed as the reference arm: each step = the oracle on a bounded sample of the
    workload, enough sequences that their (sequence, kv head) tasks occupy every host core
    twice over (the oracle's OpenMP loop runs over those tasks)."""
    if rank != 0:
        return None
    import oracle
    from paged_kv_cache_290_gb300 import workloads as W
    oracle.build()
    b = W.WORKLOADS[args.workload](keep_contiguous=False, keep_pre=False)
    sp = 0 if args.no_shared_prefix else shared_prefix_tokens(b)
    threads = oracle.get_threads()
    g = torch.Generator().manual_seed(11)
    order = [i for i in torch.randperm(b.num_seqs, generator=g).tolist()
             if b.seqs[i].query_len > 0]
    per_step = max(1, min(len(order), -(-2 * threads // b.num_kv_heads)))
    sample = lambda i: [order[(i * per_step + j) % len(order)] for j in range(per_step)]
    for i in range(args.warmup):
        _oracle_sample_seconds(b, sample(i))
    times, bytes_ = [], []
    for i in range(args.steps):
        seqs = sample(args.warmup + i)
        times.append(_oracle_sample_seconds(b, seqs))
        bytes_.append(_sample_bytes(b, seqs))
    total_t = sum(times)
    value = sum(bytes_) / total_t / 1e9
    return {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_t * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_config(args.workload, b, sp, world),
        "impl": "reference",
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"attention of {per_step} sequences of the workload per step "
                                   f"({per_step * b.num_kv_heads} (sequence, kv head) tasks "
                                   f"for {threads} cores; all their rows and heads), cycling "
                                   f"through the batch; fp64 C oracle with OpenMP"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-shared-prefix", action="store_true",
                    help="attend an aliased prefix per sequence instead of once for all rows")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--extra-cpu-seconds", type=float, default=4.0,
                    help="oracle budget of each extra workload's CPU baseline")
    ap.add_argument("--soak-seconds", type=float, default=1.5,
                    help="back-to-back steps after the timed region, for the clock sampler")
    ap.add_argument("--no-workloads", action="store_true",
                    help="measure only --workload (the default line also measures the other "
                         "workloads of the task's configurations)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    try:
        res = run_ours(args, world, rank, local)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

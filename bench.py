"""Benchmark of the paged-attention hot path on one GB300 (or N replicas).

Headline workload: the GQA decode batch with the Llama-3-8B attention shape
(64 requests x 1 query, seq_lens U[128, 4096], 32 q / 8 kv heads, head_size
128, block_size 16, bf16).  One step = the whole decode hot path on that
batch: the cache write of the step's 64 new tokens, split-KV stage 1 with the
split count of the library's planner, and the LSE merge.  ``value`` is decode KV throughput in
GB/s: the bytes of K and V the step must read (4096 B per token per kv-head
pair, summed over the batch) divided by the time per step.

Secondary lines in the same JSON record (same kernels, timed alone): the
chunked-prefill workload (TFLOP/s of causal-visible work), the long-context
split-KV decode (Llama-3-70B shape, 8 x 131072), and MLA latent decode
(DeepSeek-V3 shape).

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload instead (the only other place this script runs the oracle).
Multi-GPU: ``torchrun --nproc-per-node N bench.py --gpus N`` runs N
independent replicas (weak scaling; the path has no exchange step).
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
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "decode KV GB/s (% HBM peak); prefill TFLOP/s (% bf16 peak); 1 GB300"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained",
                                                     p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK, source="fallback")


def kernel_source_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_50_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary_name, sha):
    """DRAM bytes per launch recorded by an ncu capture of this kernel source
    (``traffic_bytes_per_launch`` and ``source_sha`` lines in the summary under
    profiles/); None if absent or if the kernel changed since."""
    path = os.path.join(ROOT, "profiles", summary_name)
    try:
        text = open(path).read()
    except OSError:
        return None
    m_sha = re.search(r"source_sha:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != sha:
        return None
    return float(m_tr.group(1))


class ClockSampler:
    """nvidia-smi clock/throttle samples while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "10"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class NvmlClockSampler:
    """SM clock and throttle reasons polled through NVML from a host thread
    every ~0.5 ms, so that samples land inside a timed region of a few
    milliseconds; the device is matched to the CUDA device by UUID.  Falls
    back to ClockSampler (nvidia-smi, 10 ms) where NVML cannot be loaded."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        import ctypes
        import threading
        self.ct, self.threading = ctypes, threading
        self.dev = device_index
        self.samples = []            # (perf_counter, sm MHz, reason bits)
        self.windows = []            # (t0, t1) of timed regions
        self.fallback = None
        self.nvml = self.handle = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = ctypes.c_void_p()
            uuid = str(getattr(torch.cuda.get_device_properties(device_index), "uuid", ""))
            ok = False
            if uuid:
                ok = nv.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) == 0
            if not ok and nv.nvmlDeviceGetHandleByIndex_v2(device_index, ctypes.byref(h)) != 0:
                raise OSError("no NVML handle")
            self.nvml, self.handle = nv, h
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(
                h, 1, ctypes.byref(mx)) == 0 else None
            self._reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        except (OSError, AttributeError):
            self.fallback = ClockSampler(device_index)

    def _poll(self):
        ct, nv, h = self.ct, self.nvml, self.handle
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) == 0:
                r = rs.value if self._reasons(h, ct.byref(rs)) == 0 else 0
                self.samples.append((time.perf_counter(), float(clk.value), int(r)))
            time.sleep(0.0005)

    def start(self):
        if self.fallback is not None:
            return self.fallback.start()
        self._stop = self.threading.Event()
        self._thread = self.threading.Thread(target=self._poll, daemon=True)
        self._thread.start()
        while not self.samples and self._thread.is_alive():
            time.sleep(0.001)

    def mark(self, t0, t1):
        self.windows.append((t0, t1))

    def stop(self):
        if self.fallback is not None:
            return self.fallback.stop()
        self._stop.set()
        self._thread.join()
        inside = [x for x in self.samples if any(a <= x[0] <= b for a, b in self.windows)]
        use = inside or self.samples
        reasons = sorted({name for _, _, r in use for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(x[1] for x in use) if use else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(use),
                "samples_in_timed_regions": len(inside), "timed_regions": len(self.windows),
                "how": "NVML from a host thread every ~0.5 ms; the median over samples taken "
                       "inside the timed regions (all samples if none landed)"}


def max_over_ranks(values, dist=None, device=None):
    """Element-wise maximum of this rank's timings (a list of floats) over the
    process group -- the slowest replica sets the job's time; unchanged on a
    single process."""
    if dist is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def replica_rate(world, bytes_per_step, steps, seconds):
    """Whole-job GB/s of `world` replicas that each moved bytes_per_step per
    step for `steps` steps in `seconds` (the slowest rank's time)."""
    return world * bytes_per_step * steps / seconds / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def to_dev_bf16(bits, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(
        torch.bfloat16)


def to_dev(a, dtype, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


# ---------------------------------------------------------------------------
# Headline: GQA decode step (cache write + split-KV stage 1 + LSE merge).
# ---------------------------------------------------------------------------

class DecodeStep:
    def __init__(self, pa, b, device, n_pools=4):
        self.pa, self.b, self.device = pa, b, device
        N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
        base = to_dev_bf16(b.pool, device)
        # Several copies of the pool so that consecutive steps never find the
        # previous step's K/V in L2 (4 x 0.53 GB >> 129 MB of L2).
        self.pools = [base] + [base.clone() for _ in range(n_pools - 1)]
        self.q = to_dev_bf16(b.q, device).view(N, hq, d)
        self.key = to_dev_bf16(b.key, device)
        self.value = to_dev_bf16(b.value, device)
        self.slots = to_dev(b.slot_mapping, torch.int64, device)
        self.table = to_dev(b.block_table, torch.int32, device)
        self.seq = to_dev(b.seq_lens, torch.int32, device)
        self.max_seq = int(b.seq_lens.max())
        # The library's decode planner (about twelve CTAs per SM, never more
        # splits than the page's rule): 4 for this batch, where the page's
        # rule gives 8 and each extra CTA costs start-up and combine time.
        self.S = pa.pa_decode_num_kv_splits(N, b.num_kv_heads, self.max_seq,
                                            pa.pa_device_sm_count())
        self.S_page = pa.pa_num_kv_splits(self.max_seq, pa.pa_device_sm_count())
        self.ws = pa.decode_workspace(N, hq, self.S, d, device=device)
        self.out = torch.empty((N, hq, d), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((N, hq), dtype=torch.float32, device=device)

    def run(self, k, ev=None):
        pa, pool = self.pa, self.pools[k % len(self.pools)]
        pa.pa_reshape_and_cache(self.key, self.value, pool, self.slots)
        if ev is not None:
            ev[0].record()
        pa.pa_decode_splitkv(self.q, pool, self.table, self.seq, self.b.scale, self.ws,
                             self.max_seq)
        if ev is not None:
            ev[1].record()
        pa.pa_lse_merge(self.ws, self.out, self.lse)


def run_e2e(pa, b, step, steps, warmup, device):
    """Same step through the public API with the step's inputs in pinned host
    memory: every step copies q / new K,V / slot_mapping / block_table /
    seq_lens host -> device, makes the three calls, and reads out + lse back
    device -> host.  As a serving loop would, the copies run beside the
    compute: while step k computes, a second stream brings in step k + 1's
    inputs and sends back step k - 1's result (device buffers alternate
    between steps), and the host waits for step k - 1's result only after
    step k is enqueued.  The timed region includes the first step's input
    copy and the last step's result copy."""
    N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
    # The step's inputs travel as one packed transfer and its results as
    # another: q, the new K and V, slots, block table and lengths at
    # 256-byte-aligned offsets of one pinned buffer, copied into one device
    # buffer of which the library's arguments are views; out and LSE likewise
    # in one device buffer, read back whole.
    parts = [("q", b.q.view(np.int16), torch.bfloat16, (N, hq, d)),
             ("key", b.key.view(np.int16), torch.bfloat16, b.key.shape),
             ("value", b.value.view(np.int16), torch.bfloat16, b.value.shape),
             ("slots", b.slot_mapping, torch.int64, b.slot_mapping.shape),
             ("table", b.block_table, torch.int32, b.block_table.shape),
             ("seq", b.seq_lens, torch.int32, b.seq_lens.shape)]
    align = lambda x: (x + 255) // 256 * 256
    offs, total = {}, 0
    for name, arr, _, _ in parts:
        offs[name] = total
        total = align(total + arr.nbytes)
    hbuf = torch.empty(total, dtype=torch.uint8).pin_memory()
    for name, arr, _, _ in parts:
        o = offs[name]
        hbuf[o:o + arr.nbytes].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8).reshape(-1)))
    o_bytes, l_bytes = N * hq * d * 2, N * hq * 4
    nbuf = len(step.pools)
    dbufs = [torch.empty(total, dtype=torch.uint8, device=device) for _ in range(nbuf)]
    obufs = [torch.empty(align(o_bytes) + l_bytes, dtype=torch.uint8, device=device)
             for _ in range(nbuf)]
    res_h = [torch.empty(obufs[0].numel(), dtype=torch.uint8).pin_memory() for _ in range(nbuf)]
    h2d, d2h = total, obufs[0].numel()

    def bind(k):
        j = k % nbuf
        for name, arr, dt, shape in parts:
            o = offs[name]
            setattr(step, name, dbufs[j][o:o + arr.nbytes].view(dt).view(*shape))
        step.out = obufs[j][:o_bytes].view(torch.bfloat16).view(N, hq, d)
        step.lse = obufs[j][align(o_bytes):].view(torch.float32).view(N, hq)

    copy_stream = torch.cuda.Stream(device=device)

    def enqueue(k):
        # Step k's compute; beside it, step k + 1's inputs in and step k - 1's
        # result out.  The fork and join events order both against the
        # compute stream's earlier and later work.
        main = torch.cuda.current_stream()
        fork, join = torch.cuda.Event(), torch.cuda.Event()
        fork.record(main)
        copy_stream.wait_event(fork)
        with torch.cuda.stream(copy_stream):
            dbufs[(k + 1) % nbuf].copy_(hbuf, non_blocking=True)
            res_h[(k - 1) % nbuf].copy_(obufs[(k - 1) % nbuf], non_blocking=True)
        join.record(copy_stream)
        bind(k)
        step.run(k)
        main.wait_event(join)

    def prologue():
        dbufs[0].copy_(hbuf, non_blocking=True)

    def epilogue(n):
        res_h[(n - 1) % nbuf].copy_(obufs[(n - 1) % nbuf], non_blocking=True)

    # One CUDA graph per pool copy (the steps cycle through nbuf buffer sets),
    # replayed; if capture is not possible, the same work is issued call by
    # call.
    prologue()
    for k in range(warmup):
        enqueue(k)
    torch.cuda.synchronize()
    launch = "cuda graph per step"
    graphs = []
    try:
        for k in range(nbuf):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                enqueue(k)
            graphs.append(g)
        prologue()
        for g in graphs:
            g.replay()
        torch.cuda.synchronize()
    except RuntimeError:
        graphs, launch = [], "eager"
        torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    done = [torch.cuda.Event() for _ in range(nbuf)]

    def run(n):
        prologue()
        for k in range(n):
            if graphs:
                graphs[k % nbuf].replay()
            else:
                enqueue(k)
            done[k % nbuf].record(stream)
            if k >= 1:
                done[(k - 1) % nbuf].synchronize()   # step k - 2's result is home
        epilogue(n)
        stream.synchronize()

    run(warmup)
    t0 = time.perf_counter()
    run(steps)
    dt = time.perf_counter() - t0
    return dt, h2d, d2h, (launch + ", one packed copy each way on a second stream beside the "
                          "compute (step k+1's inputs in and step k-1's result out while step k "
                          "computes), step k+1 enqueued before the host waits")


def cpu_baseline_sample(b, budget_s=12.0, threads=None):
    """The oracle, as it stands, on a bounded sample of the decode batch: the
    whole batch once (which is also the reference of the headline's parity
    pass), then groups of requests in order until ~budget_s of CPU work.
    Returns (GB/s of KV processed, threads, sample description, (out, lse)
    of the whole batch)."""
    import oracle
    threads = threads or (os.cpu_count() or 1)
    pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    per_tok = b.num_kv_heads * b.head_size * 2 * 2
    t0 = time.perf_counter()
    ref = oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc, b.seq_lens, b.scale,
                                 threads=threads)
    elapsed = time.perf_counter() - t0
    done_bytes, n = int(b.seq_lens.astype(np.int64).sum()) * per_tok, b.num_seqs
    group = max(1, threads)
    while elapsed < budget_s:
        # A group of requests per call (so the oracle's threads have work),
        # cycling through the batch until the time budget is spent.
        grp = [(n + j) % b.num_seqs for j in range(group)]
        mask = np.zeros(b.num_tokens, np.uint8)
        mask[grp] = 1
        t0 = time.perf_counter()
        oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc, b.seq_lens, b.scale,
                               row_mask=mask, threads=threads)
        elapsed += time.perf_counter() - t0
        done_bytes += int(b.seq_lens[grp].astype(np.int64).sum()) * per_tok
        n += len(grp)
    return done_bytes / elapsed / 1e9, threads, (
        f"oracle decode attention (fp64, paged gather + softmax), {n} request-decodes cycling "
        f"through the {b.num_seqs}-request GQA decode batch, {elapsed:.1f} s of {threads} "
        "threads"), ref


# ---------------------------------------------------------------------------
# Secondary workloads: every other named configuration, its kernels timed
# alone (CUDA events on the launch stream, median of >= 50 launches), each
# line with its seed, one parity pass against the oracle on the same seeded
# inputs (the rows / requests it names), the oracle's own rate on that
# sample, and the roofline of its dominant kernel.
# ---------------------------------------------------------------------------

SECONDARY_REPS = 50
OUT_ATOL, LSE_ATOL = 1e-2, 1e-3


def time_events(fn, reps, warmup=3):
    for _ in range(warmup):
        fn()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        e0.record()
        fn()
        e1.record()
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)   # ms


def _timed_rotating(fns, reps, warmup=3):
    """Median of reps event-timed launches that cycle through fns, each bound
    to its own copy of the inputs: every pool is larger than L2, so a launch
    finds none of its pool in L2 (the copy it reads was last touched a whole
    pool's worth of traffic earlier) and no dirty lines left by a flush."""
    for k in range(warmup * len(fns)):
        fns[k % len(fns)]()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    torch.cuda.synchronize()
    for k, (e0, e1) in enumerate(evs):
        e0.record()
        fns[k % len(fns)]()
        e1.record()
    torch.cuda.synchronize()
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs)   # ms


def l2_flusher(device):
    buf = torch.empty(256 << 20, dtype=torch.uint8, device=device)
    return lambda: buf.fill_(1)


def _timed_with_flush(fn, flush, reps):
    """Median of reps event-timed launches, L2 flushed before each."""
    for _ in range(3):
        flush()
        fn()
    times = []
    for _ in range(reps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return statistics.median(times)


def _bf16_ulp(x):
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def parity(got_o, ref_o, got_l, ref_l, checked):
    """Max abs errors of a parity pass and whether every element met the
    tolerance: bf16 outputs within max(1e-2, one bf16 ulp of the oracle
    value), LSE within 1e-3 (and -inf exactly where the oracle's is)."""
    got_o, ref_o = np.asarray(got_o, np.float64), np.asarray(ref_o, np.float64)
    got_l, ref_l = np.asarray(got_l, np.float64), np.asarray(ref_l, np.float64)
    eo = np.abs(got_o - ref_o)
    bad_o = int((eo > np.maximum(OUT_ATOL, _bf16_ulp(ref_o))).sum()) + int(
        (~np.isfinite(got_o)).sum())
    fin = np.isfinite(ref_l)
    el = np.abs(got_l[fin] - ref_l[fin])
    bad_l = int((el > LSE_ATOL).sum()) + int((np.isneginf(got_l) != np.isneginf(ref_l)).sum())
    return {"max_abs_out_err": float(eo.max()) if eo.size else 0.0,
            "max_abs_lse_err": float(el.max()) if el.size else 0.0,
            "out_beyond_tol": bad_o, "lse_beyond_tol": bad_l, "pass": bad_o == 0 and bad_l == 0,
            "checked": checked,
            "tolerance": "out: max(1e-2, 1 bf16 ulp of the oracle value); lse: 1e-3"}


def _timed_oracle(fn):
    t0 = time.perf_counter()
    r = fn()
    return r, time.perf_counter() - t0


def cpu_line(rate, unit, seconds, threads, sample):
    return {"value": rate, "unit": unit, "cores": threads, "kind": "oracle",
            "sample": f"{sample}; {seconds:.2f} s of {threads} threads"}


def roofline(bound, achieved, pk, unit, kernel, algo, traffic=None):
    if bound == "hbm":
        peak, src = pk["hbm_gbs"], "MEASURED_PEAKS hbm_gbs"
    else:
        peak, src = pk["bf16_tflops"], "MEASURED_PEAKS bf16_tflops (burst)"
    if pk["source"] != "measured":
        src = "fallback"
    return {"bound": bound, "kernel": kernel, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic, "algorithmic_per_launch": algo,
            "peak_source": src + (" (of measured)" if pk["source"] == "measured" else
                                  " (of fallback)")}


def sub_pool(pool, block_table, seq_lens, reqs):
    """The blocks of requests ``reqs`` gathered into a small pool, with a
    table that numbers them 0, 1, ... in request order: the oracle then runs
    on those requests alone (the whole pool in fp64 can take tens of GB)."""
    bs = pool.shape[2] if pool.ndim == 5 else pool.shape[1]
    ids = [block_table[r, :(int(seq_lens[r]) + bs - 1) // bs] for r in reqs]
    width = max(1, max(len(x) for x in ids))
    table = np.full((len(reqs), width), -1, np.int32)
    k = 0
    for i, x in enumerate(ids):
        table[i, :len(x)] = np.arange(k, k + len(x), dtype=np.int32)
        k += len(x)
    return pool[np.concatenate(ids)], table


def _new_slots(table, seq_lens, reqs, bs):
    """Slots of each request's newest token (position seq_len - 1) in the
    small pool of sub_pool."""
    return np.array([int(table[k, (int(seq_lens[r]) - 1) // bs]) * bs + (int(seq_lens[r]) - 1) % bs
                     for k, r in enumerate(reqs)], np.int64)


def _last_rows(b):
    return b.query_start_loc[1:] - 1


def bench_tiny(pa, device, pk, flush, reps=SECONDARY_REPS, check=True):
    """The tiny paged-attention batch: the whole step (cache write + varlen
    attention with LSE), launch-bound; timed warm (everything fits in L2)."""
    b = workloads.tiny_paged()
    pool = to_dev_bf16(b.pool, device)
    q, key, val = (to_dev_bf16(x, device) for x in (b.q, b.key, b.value))
    slots = to_dev(b.slot_mapping, torch.int64, device)
    table = to_dev(b.block_table, torch.int32, device)
    qsl = to_dev(b.query_start_loc, torch.int32, device)
    seq = to_dev(b.seq_lens, torch.int32, device)
    out = torch.empty_like(q)
    lse = torch.empty((b.num_tokens, b.num_q_heads), dtype=torch.float32, device=device)
    mq = int(b.query_lens.max())

    def step():
        pa.pa_reshape_and_cache(key, val, pool, slots)
        pa.pa_varlen_fwd(q, pool, table, qsl, seq, mq, b.scale, out=out, lse=lse)
    ms = time_events(step, reps)
    tf = b.causal_flops() / (ms * 1e-3) / 1e12
    res = {"workload": b.name, "seed": b.seed, "kernels": "reshape_and_cache + varlen_tc_kernel",
           "ms": ms, "reps": reps, "tflops": tf, "causal_flops": b.causal_flops(),
           "l2": "warm (the whole batch is 170 KB)",
           "note": "launch-bound: 7 query rows; the time is two kernel launches"}
    if check:
        import oracle
        ref_pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
        (ro, rl), dt = _timed_oracle(lambda: oracle.paged_attention(
            b.q, ref_pool, b.block_table, b.query_start_loc, b.seq_lens, b.scale))
        res["parity"] = parity(out.float().cpu().numpy(), ro, lse.cpu().numpy(), rl,
                               "all 7 rows x 4 heads")
        res["parity"]["cache_write_bit_exact"] = bool(np.array_equal(
            pool.view(torch.int16).cpu().numpy().view(np.uint16), ref_pool))
        res["cpu_baseline"] = cpu_line(b.causal_flops() / dt / 1e12, "TFLOP/s", dt,
                                       oracle.default_threads(),
                                       "oracle varlen attention over the whole tiny batch")
    return res


def bench_prefill(pa, device, pk, flush, reps=SECONDARY_REPS, check=True):
    """Chunked prefill: the varlen kernel on its own, L2 flushed before each
    launch."""
    b = workloads.chunked_prefill()
    pool = to_dev_bf16(b.pool, device)
    q = to_dev_bf16(b.q, device)
    pa.pa_reshape_and_cache(to_dev_bf16(b.key, device), to_dev_bf16(b.value, device), pool,
                            to_dev(b.slot_mapping, torch.int64, device))
    table = to_dev(b.block_table, torch.int32, device)
    qsl = to_dev(b.query_start_loc, torch.int32, device)
    seq = to_dev(b.seq_lens, torch.int32, device)
    out = torch.empty_like(q)
    lse = torch.empty((b.num_tokens, b.num_q_heads), dtype=torch.float32, device=device)
    mq = int(b.query_lens.max())

    def prefill():
        pa.pa_varlen_fwd(q, pool, table, qsl, seq, mq, b.scale, out=out, lse=lse)
    ms = _timed_with_flush(prefill, flush, reps)
    warm = time_events(prefill, reps)
    tf = b.causal_flops() / (ms * 1e-3) / 1e12
    res = {"workload": b.name, "seed": b.seed, "kernel": "varlen_tc_kernel", "ms": ms,
           "warm_ms": warm, "reps": reps, "tflops": tf, "causal_flops": b.causal_flops(),
           "frac_of_bf16_peak": tf / pk["bf16_tflops"],
           "l2": "flushed (256 MB write) before each launch",
           "roofline": roofline("tensor", tf, pk, "TFLOP/s", "varlen_tc_kernel",
                                b.causal_flops(),
                                profiled_traffic("varlen_tc_chunked_prefill.md",
                                                 kernel_source_sha(["varlen_tc.cu",
                                                                    "tc_common.cuh"])))}
    if check:
        import oracle
        prefill()
        torch.cuda.synchronize()
        rng = np.random.default_rng(1003)
        mask = np.zeros(b.num_tokens, np.uint8)
        for i in range(b.num_seqs):
            a, e = int(b.query_start_loc[i]), int(b.query_start_loc[i + 1])
            mask[[a, e - 1]] = 1
            mask[rng.integers(a, e, size=2)] = 1
        rows = mask.astype(bool)
        ref_pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
        (ro, rl), dt = _timed_oracle(lambda: oracle.paged_attention(
            b.q, ref_pool, b.block_table, b.query_start_loc, b.seq_lens, b.scale, row_mask=mask))
        res["parity"] = parity(out.float().cpu().numpy()[rows], ro[rows],
                               lse.cpu().numpy()[rows], rl[rows],
                               f"{int(rows.sum())} rows (first, last and 2 random of each "
                               f"request) x {b.num_q_heads} heads")
        # Causal-visible flops of the sampled rows.
        pos = np.concatenate([np.arange(int(b.seq_lens[i] - b.query_lens[i]), int(b.seq_lens[i]))
                              for i in range(b.num_seqs)])
        fl = 4 * b.head_size * b.num_q_heads * int((pos[rows] + 1).sum())
        res["cpu_baseline"] = cpu_line(fl / dt / 1e12, "TFLOP/s", dt, oracle.default_threads(),
                                       f"oracle varlen attention on the {int(rows.sum())} "
                                       "sampled rows")
    del pool, q, out
    torch.cuda.empty_cache()
    return res


def _decode_check(b, out, lse, reqs, ref_fn, unit_bytes):
    """Parity of decode outputs on requests ``reqs`` and the oracle's rate
    on them: ref_fn() -> (out, lse) of those requests, in order."""
    import oracle
    (ro, rl), dt = _timed_oracle(ref_fn)
    par = parity(out.float().cpu().numpy()[reqs], ro, lse.cpu().numpy()[reqs], rl,
                 f"requests {[int(r) for r in reqs]} (all heads)")
    done = int(b.seq_lens[reqs].astype(np.int64).sum()) * unit_bytes
    return par, cpu_line(done / dt / 1e9, "GB/s", dt, oracle.default_threads(),
                         f"oracle decode on the {len(reqs)} checked requests")


def bench_long_decode(pa, device, pk, flush, reps=SECONDARY_REPS, check=True):
    """Long-context split-KV decode (8 x 131072): stage 1, and stage 1 +
    merge, cycling through two pool copies."""
    b = workloads.long_decode()
    N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
    pool = to_dev_bf16(b.pool, device)
    pa.pa_reshape_and_cache(to_dev_bf16(b.key, device), to_dev_bf16(b.value, device), pool,
                            to_dev(b.slot_mapping, torch.int64, device))
    q = to_dev_bf16(b.q, device).view(N, hq, d)
    table, seq = to_dev(b.block_table, torch.int32, device), to_dev(b.seq_lens, torch.int32,
                                                                    device)
    S = pa.pa_num_kv_splits(131072, pa.pa_device_sm_count())
    ws = pa.decode_workspace(N, hq, S, d, device=device)
    o = torch.empty((N, hq, d), dtype=torch.bfloat16, device=device)
    lo = torch.empty((N, hq), dtype=torch.float32, device=device)
    pools = [pool, pool.clone()]
    stage1 = [lambda p=p: pa.pa_decode_splitkv(q, p, table, seq, b.scale, ws, 131072)
              for p in pools]
    st1 = _timed_rotating(stage1, reps)
    warm = time_events(stage1[0], reps)
    both = _timed_rotating([lambda p=p: pa.pa_decode(q, p, table, seq, b.scale, ws, o, lo, 131072)
                            for p in pools], reps)
    gbs = b.kv_bytes() / (st1 * 1e-3) / 1e9
    sha = kernel_source_sha(["decode.cu", "pa_common.cuh"])
    res = {"workload": b.name, "seed": b.seed, "num_splits": S, "stage1_ms": st1,
           "stage1_warm_ms": warm, "reps": reps, "decode_plus_merge_ms": both,
           "kv_bytes": b.kv_bytes(), "stage1_gbs": gbs, "frac_of_hbm_peak": gbs / pk["hbm_gbs"],
           "step_gbs": b.kv_bytes() / (both * 1e-3) / 1e9, "l2": "2 rotating pool copies",
           "roofline": roofline("hbm", gbs, pk, "GB/s", "decode_splitkv_kernel", b.kv_bytes(),
                                profiled_traffic("decode_splitkv_long_decode.md", sha))}
    if check:
        import oracle
        pa.pa_decode(q, pools[0], table, seq, b.scale, ws, o, lo, 131072)
        torch.cuda.synchronize()
        reqs = np.array([0, 5])

        def ref():
            sp, st = sub_pool(b.pool, b.block_table, b.seq_lens, reqs)
            sp = oracle.reshape_and_cache(b.key[reqs], b.value[reqs], sp,
                                          _new_slots(st, b.seq_lens, reqs, b.block_size),
                                          b.block_size)
            return oracle.paged_attention(b.q[_last_rows(b)[reqs]], sp, st,
                                          np.arange(len(reqs) + 1, dtype=np.int32),
                                          b.seq_lens[reqs], b.scale)
        res["parity"], res["cpu_baseline"] = _decode_check(b, o, lo, reqs, ref,
                                                           b.num_kv_heads * d * 2 * 2)
    del pool, pools, q, ws
    torch.cuda.empty_cache()
    return res


def bench_mla(pa, device, pk, flush, reps=SECONDARY_REPS, check=True):
    """MLA latent decode (DeepSeek-V3 shape), split count from the library's
    planner, cycling through two pool copies; the step's cache write of the
    128 new latent rows timed alone."""
    m = workloads.mla_decode()
    pool = to_dev_bf16(m.pool, device)
    q = to_dev_bf16(m.q, device)
    table, seq = to_dev(m.block_table, torch.int32, device), to_dev(m.seq_lens, torch.int32,
                                                                    device)
    mx = int(m.seq_lens.max())
    S = pa.pa_mla_num_kv_splits(m.batch, m.num_heads, mx, pa.pa_device_sm_count())
    ws = pa.decode_workspace(m.batch, m.num_heads, S, m.kv_lora_rank, device=device)
    o = torch.empty((m.batch, m.num_heads, m.kv_lora_rank), dtype=torch.bfloat16, device=device)
    lo = torch.empty((m.batch, m.num_heads), dtype=torch.float32, device=device)
    pools = [pool, pool.clone()]
    mla = [lambda p=p: pa.pa_mla_decode(q, p, table, seq, m.scale, ws, o, lo, max_seq_len=mx)
           for p in pools]
    ms = _timed_rotating(mla, reps)
    warm = time_events(mla[0], reps)
    kv_c, k_pe, slots = workloads.mla_new_tokens(m)
    d_kv_c, d_k_pe = to_dev_bf16(kv_c, device), to_dev_bf16(k_pe, device)
    d_slots = to_dev(slots, torch.int64, device)
    scratch = pools[1]
    write_ms = _timed_with_flush(lambda: pa.pa_mla_cache_write(d_kv_c, d_k_pe, scratch, d_slots),
                                 flush, reps)
    gbs = m.kv_bytes() / (ms * 1e-3) / 1e9
    flops = int(m.seq_lens.astype(np.int64).sum()) * m.num_heads * 2 * (
        m.kv_lora_rank + m.rope_dim + m.kv_lora_rank)
    sha = kernel_source_sha(["mla_tc.cu", "tc_common.cuh"])
    res = {"workload": m.name, "seed": m.seed, "num_splits": S,
           "splits_from": "pa_mla_num_kv_splits", "ms": ms, "warm_ms": warm, "reps": reps,
           "kv_bytes": m.kv_bytes(), "gbs": gbs, "frac_of_hbm_peak": gbs / pk["hbm_gbs"],
           "tflops": flops / (ms * 1e-3) / 1e12,
           "cache_write_us": write_ms * 1e3, "cache_write_tokens": int(m.batch),
           "l2": "2 rotating pool copies (cache write: L2 flushed)",
           "roofline": roofline("hbm", gbs, pk, "GB/s", "mla_tc_kernel", m.kv_bytes(),
                                profiled_traffic("mla_tc_mla_decode.md", sha))}
    if check:
        import oracle
        mla[0]()
        torch.cuda.synchronize()
        order = np.argsort(m.seq_lens, kind="stable")
        rng = np.random.default_rng(1005)
        pick = set(order[:2].tolist()) | set(order[-2:].tolist()) | set(
            rng.choice(m.batch, 4, replace=False).tolist())
        reqs = np.array(sorted(pick))
        mask = np.zeros(m.batch, np.uint8)
        mask[reqs] = 1

        def ref():
            ro, rl = oracle.mla_decode(m.q, m.pool, m.block_table, m.seq_lens, m.scale,
                                       req_mask=mask)
            return ro[reqs], rl[reqs]
        res["parity"], res["cpu_baseline"] = _decode_check(
            m, o, lo, reqs, ref, (m.kv_lora_rank + m.rope_dim) * 2)
    del pool, pools, q, ws
    torch.cuda.empty_cache()
    return res


def bench_mla_prefill(pa, device, pk, flush, reps=SECONDARY_REPS, check=True):
    """MLA chunked prefill, multi-head formulation (DeepSeek-V3 shape): the
    kv_b_proj expansion of every context token and the attention over the
    expanded keys and values, timed together and apart."""
    m = workloads.mla_prefill()
    pool = to_dev_bf16(m.pool, device)
    pa.pa_mla_cache_write(to_dev_bf16(m.kv_c, device), to_dev_bf16(m.k_pe, device), pool,
                          to_dev(m.slot_mapping, torch.int64, device))
    q = to_dev_bf16(m.q, device)
    wt = to_dev_bf16(m.w_kv_b, device)
    table = to_dev(m.block_table, torch.int32, device)
    qsl = to_dev(m.query_start_loc, torch.int32, device)
    seq = to_dev(m.seq_lens, torch.int32, device)
    S = int(m.seq_lens.max())
    mq = int(m.query_lens.max())
    ws = torch.empty(pa.pa_mla_prefill_workspace_bytes(m.num_seqs, S, m.num_heads),
                     dtype=torch.uint8, device=device)
    out = torch.empty((m.num_tokens, m.num_heads, 128), dtype=torch.bfloat16, device=device)
    lse = torch.empty((m.num_tokens, m.num_heads), dtype=torch.float32, device=device)
    kv_elems = m.num_seqs * S * m.num_heads
    k_ws = ws[:kv_elems * 192 * 2].view(torch.bfloat16).view(m.num_seqs, S, m.num_heads, 192)
    v_ws = ws[kv_elems * 192 * 2:kv_elems * 320 * 2].view(torch.bfloat16).view(
        m.num_seqs, S, m.num_heads, 128)

    def call():
        pa.pa_mla_prefill(q, pool, wt, table, qsl, seq, mq, m.scale, ws, S, out=out, lse=lse)
    total = _timed_with_flush(call, flush, reps)
    warm = time_events(call, reps)
    expand = _timed_with_flush(lambda: pa.pa_mla_expand_kv(pool, wt, table, seq, k_ws, v_ws),
                               flush, reps)
    attn = total - expand
    ef, af = m.expand_flops(), m.causal_flops()
    tf = (ef + af) / (total * 1e-3) / 1e12
    res = {"workload": m.name, "seed": m.seed, "ms": total, "warm_ms": warm, "reps": reps,
           "expand_ms": expand, "attention_ms": attn,
           "expand_tflops": ef / (expand * 1e-3) / 1e12,
           "attention_tflops": af / (attn * 1e-3) / 1e12,
           "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"],
           "expanded_bytes": kv_elems * 320 * 2,
           "l2": "flushed (256 MB write) before each launch",
           "roofline": roofline("tensor", tf, pk, "TFLOP/s",
                                "mla_expand_kernel + varlen_tc_kernel", ef + af)}
    if check:
        import oracle
        call()
        torch.cuda.synchronize()
        ref_pool = oracle.mla_cache_write(m.kv_c, m.k_pe, m.pool, m.slot_mapping, m.block_size)
        rng = np.random.default_rng(1007)
        rows = np.zeros(m.num_tokens, np.uint8)
        for i in range(m.num_seqs):
            a, e = int(m.query_start_loc[i]), int(m.query_start_loc[i + 1])
            rows[[a, e - 1]] = 1
            rows[rng.integers(a, e)] = 1
        heads = np.zeros(m.num_heads, np.uint8)
        heads[rng.choice(m.num_heads, 8, replace=False)] = 1
        (ro, rl), dt = _timed_oracle(lambda: oracle.mla_prefill(
            m.q, ref_pool, m.w_kv_b, m.block_table, m.query_start_loc, m.seq_lens, m.scale,
            head_mask=heads, row_mask=rows))
        r, h = rows.astype(bool), heads.astype(bool)
        res["parity"] = parity(out.float().cpu().numpy()[r][:, h], ro[r][:, h],
                               lse.cpu().numpy()[r][:, h], rl[r][:, h],
                               f"{int(r.sum())} rows x {int(h.sum())} heads")
        pos = np.concatenate([np.arange(int(m.seq_lens[i] - m.query_lens[i]), int(m.seq_lens[i]))
                              for i in range(m.num_seqs)])
        fl = 2 * (192 + 128) * int(h.sum()) * int((pos[r] + 1).sum())
        res["cpu_baseline"] = cpu_line(fl / dt / 1e12, "TFLOP/s", dt, oracle.default_threads(),
                                       "oracle MLA prefill on the checked rows x heads "
                                       "(rate counts their causal-visible attention flops; the "
                                       "oracle's time also holds its kv_b_proj expansion)")
    del pool, q, wt, ws
    torch.cuda.empty_cache()
    return res


def fp8_kernel_name(d, grp):
    """The fp8 stage-1 instantiation the library launches: groups of more
    than 8 heads take two n-tiles (and, for d = 128, a fourth ring stage)."""
    wide = grp > 8
    stages = (4 if wide else 3) if d == 128 else 8
    return f"decode_splitkv_fp8_kernel<{d},{stages},{2 if wide else 1}>"


def bench_fp8_decode(pa, device, pk, flush, reps=SECONDARY_REPS, check=True):
    """Split-KV decode over an fp8 (e4m3) pool, on the GQA decode batch and the
    long-context batch: stage 1 alone, and the whole step (quantising cache
    write + stage 1 + merge)."""
    res = {}
    ks, vs = workloads.FP8_K_SCALE, workloads.FP8_V_SCALE
    for make in (workloads.gqa_decode, workloads.long_decode):
        b = make(with_pool=False)
        N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
        host_pool = workloads.fp8_pool(b)
        pool = torch.from_numpy(host_pool).to(device)
        q = to_dev_bf16(b.q, device).view(N, hq, d)
        key, value = to_dev_bf16(b.key, device), to_dev_bf16(b.value, device)
        slots = to_dev(b.slot_mapping, torch.int64, device)
        table = to_dev(b.block_table, torch.int32, device)
        seq = to_dev(b.seq_lens, torch.int32, device)
        mx = int(b.seq_lens.max())
        sms = pa.pa_device_sm_count()
        # The long-context batch keeps the page's rule (its workload fixes
        # S); the GQA batch takes the library's planner, as the headline.
        S = (pa.pa_num_kv_splits(mx, sms) if make is workloads.long_decode
             else pa.pa_decode_num_kv_splits(N, b.num_kv_heads, mx, sms))
        ws = pa.decode_workspace(N, hq, S, d, device=device)
        o = torch.empty((N, hq, d), dtype=torch.bfloat16, device=device)
        lo = torch.empty((N, hq), dtype=torch.float32, device=device)
        pools = [pool, pool.clone()]

        def step(p):
            pa.pa_reshape_and_cache_fp8(key, value, p, slots, ks, vs)
            pa.pa_decode_fp8(q, p, table, seq, b.scale, ks, vs, ws, o, lo, mx)
        stage1 = [lambda p=p: pa.pa_decode_splitkv_fp8(q, p, table, seq, b.scale, ks, vs, ws, mx)
                  for p in pools]
        st1 = _timed_rotating(stage1, reps)
        warm = time_events(stage1[0], reps)
        both = _timed_rotating([lambda p=p: step(p) for p in pools], reps)
        kv = b.kv_bytes() // 2                      # one byte per element
        gbs = kv / (st1 * 1e-3) / 1e9
        kname = fp8_kernel_name(d, b.num_q_heads // b.num_kv_heads)
        sha = kernel_source_sha(["decode_fp8.cu", "pa_common.cuh"])
        short = "gqa_decode" if make is workloads.gqa_decode else "long_decode"
        line = {"seed": b.seed, "pool_seed": [b.seed, 2], "num_splits": S, "stage1_ms": st1,
                "stage1_warm_ms": warm, "reps": reps, "step_ms": both, "kv_bytes": kv,
                "stage1_gbs": gbs, "frac_of_hbm_peak": gbs / pk["hbm_gbs"],
                "step_gbs": kv / (both * 1e-3) / 1e9, "kernel": kname,
                "l2": "2 rotating pool copies",
                "roofline": roofline("hbm", gbs, pk, "GB/s", kname, kv,
                                     profiled_traffic(f"decode_splitkv_fp8_{short}.md", sha))}
        if check:
            import oracle
            step(pools[0])
            torch.cuda.synchronize()
            reqs = np.array([0, 5])
            bs = b.block_size

            def ref():
                sp, st = sub_pool(host_pool, b.block_table, b.seq_lens, reqs)
                sp = oracle.reshape_and_cache_fp8(b.key[reqs], b.value[reqs], sp,
                                                  _new_slots(st, b.seq_lens, reqs, bs), bs, ks, vs)
                part = oracle.split_partials_fp8(b.q[_last_rows(b)[reqs]], sp, st,
                                                 b.seq_lens[reqs], b.scale, ks, vs, 1)
                return oracle.lse_merge(part)
            line["parity"], line["cpu_baseline"] = _decode_check(b, o, lo, reqs, ref,
                                                                 b.num_kv_heads * d * 2)
        res[b.name] = line
        del pool, pools, q, ws, host_pool
        torch.cuda.empty_cache()
    return res


def bench_cascade(pa, device, pk, flush, reps=SECONDARY_REPS, check=True):
    """Cascade attention on 64 decode requests sharing a prompt (4096 tokens:
    17 MB of K/V per layer, L2-resident; 32768 tokens: 134 MB, more than L2),
    against plain split-KV decode of the same batch, which reads the prompt
    once per request."""
    res = {}
    for prefix in (4096, 32768):
        b = workloads.shared_prefix_decode(prefix_tokens=prefix)
        N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
        pool = to_dev_bf16(b.pool, device)
        pa.pa_reshape_and_cache(to_dev_bf16(b.key, device), to_dev_bf16(b.value, device), pool,
                                to_dev(b.slot_mapping, torch.int64, device))
        q = to_dev_bf16(b.q, device)
        table = to_dev(b.block_table, torch.int32, device)
        qsl = to_dev(b.query_start_loc, torch.int32, device)
        seq = to_dev(b.seq_lens, torch.int32, device)
        P = prefix // b.block_size
        mx = int(b.seq_lens.max())
        sms = pa.pa_device_sm_count()
        S = pa.pa_num_kv_splits(mx, sms)
        ws = pa.decode_workspace(N, hq, S, d, device=device)
        S1 = pa.pa_cascade_prefix_splits(N, hq, b.num_kv_heads, prefix, sms)
        S2 = pa.pa_num_kv_splits(mx - prefix, sms)
        cws = pa.cascade_workspace(N, hq, S1, S2, d, device=device)
        o = torch.empty((N, hq, d), dtype=torch.bfloat16, device=device)
        lo = torch.empty((N, hq), dtype=torch.float32, device=device)
        plain = _timed_with_flush(lambda: pa.pa_decode(q.view(N, hq, d), pool, table, seq, b.scale,
                                                       ws, o, lo, mx), flush, reps)

        def casc_call():
            pa.pa_cascade_fwd(q, pool, table, qsl, seq, 1, P, b.scale, cws, S1, mx, out=o, lse=lo)
        casc = _timed_with_flush(casc_call, flush, reps)
        row = b.num_kv_heads * d * 2 * 2
        unique = (prefix + int((b.seq_lens - prefix).astype(np.int64).sum())) * row
        gbs = unique / (casc * 1e-3) / 1e9
        line = {"seed": b.seed, "prefix_tokens": prefix, "prefix_splits": S1,
                "suffix_splits": S2, "cascade_ms": casc, "plain_decode_ms": plain,
                "reps": reps, "speedup": plain / casc, "unique_kv_bytes": unique,
                "cascade_unique_gbs": gbs, "plain_kv_bytes": b.kv_bytes(),
                "l2": "flushed (256 MB write) before each launch",
                "roofline": roofline("hbm", gbs, pk, "GB/s",
                                     "varlen_tc_kernel (prefix) + decode_splitkv_kernel (suffix) "
                                     "+ lse_merge", unique)}
        if check:
            import oracle
            casc_call()
            torch.cuda.synchronize()
            reqs = np.array([0, 17, 63])
            rows = _last_rows(b)[reqs]
            mask = np.zeros(b.num_tokens, np.uint8)
            mask[rows] = 1
            ref_pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping,
                                                b.block_size)

            def ref():
                ro, rl = oracle.paged_attention(b.q, ref_pool, b.block_table, b.query_start_loc,
                                                b.seq_lens, b.scale, row_mask=mask)
                return ro[rows], rl[rows]
            line["parity"], line["cpu_baseline"] = _decode_check(b, o, lo, reqs, ref, row)
        res[b.name] = line
        del pool, q, ws, cws
        torch.cuda.empty_cache()
    return res


SECONDARY = {"tiny": bench_tiny, "chunked_prefill": bench_prefill,
             "long_decode": bench_long_decode, "mla_decode": bench_mla,
             "fp8_decode": bench_fp8_decode, "cascade": bench_cascade,
             "mla_prefill": bench_mla_prefill}


def secondary(pa, device, pk):
    flush = l2_flusher(device)
    return {name: fn(pa, device, pk, flush) for name, fn in SECONDARY.items()}


# ---------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["pa", "reference"], default="pa")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=sorted(SECONDARY),
                    help="time one secondary workload alone (--steps launches) and print its "
                         "record; a small command for profiler captures")
    args = ap.parse_args()
    warmup = max(3, args.warmup)
    world, rank, local = dist_env()

    if args.impl == "reference":
        return main_reference(args, warmup, world, rank)

    import paged_kv_cache_50_gb300 as pa
    from paged_kv_cache_50_gb300 import build as pa_build
    if not os.path.exists(pa.LIB_PATH):
        pa_build.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    pa.lib()
    pk = peaks()
    if args.only is not None:
        rec = SECONDARY[args.only](pa, device, pk, l2_flusher(device), reps=args.steps,
                                  check=False)
        if rank == 0:
            print(json.dumps({"only": args.only, **rec}), flush=True)
        return

    b = workloads.gqa_decode()
    step = DecodeStep(pa, b, device)
    kv_bytes = b.kv_bytes()

    clocks = NvmlClockSampler(local)
    clocks.start()
    for k in range(warmup):
        step.run(k)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    h0 = time.perf_counter()
    t_start.record()
    for k in range(args.steps):
        step.run(k)
    t_end.record()
    torch.cuda.synchronize()
    if hasattr(clocks, "mark"):
        clocks.mark(h0, time.perf_counter())
    if dist is not None:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    # The stage-1 kernel's own duration, from a second pass over the same K
    # steps with events on its stream around every stage-1 launch.  Events
    # between the step's kernels serialise their programmatic dependent
    # launches (about 8 us per step), so they stay out of the pass above.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    h0 = time.perf_counter()
    for k in range(args.steps):
        step.run(k, ev[k])
    torch.cuda.synchronize()
    if hasattr(clocks, "mark"):
        clocks.mark(h0, time.perf_counter())
    clk = clocks.stop()
    # The last step's result, for the parity pass of the oracle leg below.
    head_out, head_lse = step.out.float().cpu().numpy(), step.lse.cpu().numpy()
    dec_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    achieved = kv_bytes / (dec_ms * 1e-3) / 1e9
    sha = kernel_source_sha(["decode.cu", "pa_common.cuh"])
    traffic = profiled_traffic("decode_splitkv_gqa_decode.md", sha)

    e2e_dt, h2d, d2h, e2e_launch = run_e2e(pa, b, step, args.steps, warmup, device)
    # The job's times are the slowest replica's.
    total_ms, e2e_dt = max_over_ranks([total_ms, e2e_dt], dist, device)
    ms_per_step = total_ms / args.steps
    value = replica_rate(world, kv_bytes, args.steps, total_ms * 1e-3)
    e2e_value = replica_rate(world, kv_bytes, args.steps, e2e_dt)

    sec = None
    if not args.no_secondary and rank == 0:
        sec = secondary(pa, device, pk)

    cpu = head_parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample, (ref_o, ref_l) = cpu_baseline_sample(b)
        cpu = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
        head_parity = parity(head_out, ref_o, head_lse, ref_l,
                             f"all {b.num_seqs} requests x {b.num_q_heads} heads")

    if rank == 0:
        rec = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded numpy N(0,1) rounded to bf16; random block permutation)",
            "config": {"workload": b.name, "seed": b.seed, "num_seqs": b.num_seqs,
                       "seq_lens": "U[128,4096]",
                       "num_q_heads": 32, "num_kv_heads": 8, "head_size": 128,
                       "block_size": 16, "num_splits": step.S,
                       "splits_from": f"pa_decode_num_kv_splits (the page's rule: {step.S_page})",
                       "kv_bytes_per_step": kv_bytes,
                       "step": "cache write (64 tokens) + split-KV stage 1 + LSE merge",
                       "l2": "inputs larger than L2: 4 rotating pool copies of "
                             f"{kv_bytes / 1e9:.2f} GB", "parallelism": f"replicas x{world}",
                       "kernel_timing": "stage-1 events in a second pass of the same K steps "
                                        "(none inside the headline's timed region)"},
            "clocks": clk,
            "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "launch": e2e_launch},
            "gpu_launches": 3 * args.steps,
            "roofline": {"bound": "hbm", "kernel": "decode_splitkv_kernel<128,2,1>",
                         "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": achieved / pk["hbm_gbs"], "traffic": traffic,
                         "algorithmic_bytes_per_launch": kv_bytes,
                         "kernel_ms": dec_ms,
                         "peak_source": "MEASURED_PEAKS hbm_gbs (of measured)"
                         if pk["source"] == "measured" else "fallback 6.8 TB/s (of fallback)"},
            "cpu_baseline": cpu,
            "parity": head_parity,
            "secondary": sec,
        }
        print(json.dumps(rec), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main_reference(args, warmup, world, rank):
    """Reference arm: the fp64 oracle on the host cores, each step a bounded
    sample (8 requests) of the same GQA decode batch; rank 0 only."""
    if rank != 0:
        return
    import oracle
    b = workloads.gqa_decode()
    pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    threads = os.cpu_count() or 1
    per_tok = b.num_kv_heads * b.head_size * 2 * 2
    group = 8

    def one(k):
        first = (k * group) % b.num_seqs
        reqs = [(first + j) % b.num_seqs for j in range(group)]
        mask = np.zeros(b.num_tokens, np.uint8)
        mask[reqs] = 1
        oracle.paged_attention(b.q, pool, b.block_table, b.query_start_loc, b.seq_lens, b.scale,
                               row_mask=mask, threads=threads)
        return int(b.seq_lens[reqs].astype(np.int64).sum()) * per_tok

    for k in range(warmup):
        one(k)
    t0 = time.perf_counter()
    done = 0
    for k in range(args.steps):
        done += one(k)
    dt = time.perf_counter() - t0
    value = done / dt / 1e9
    sample = (f"fp64 oracle decode attention, {group} requests of the GQA decode batch per step "
              "(cache write done once, outside the timed region)")
    rec = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
           "steps": args.steps, "warmup": warmup, "ms_per_step": dt * 1e3 / args.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "config": {"workload": b.name, "parallelism": "host threads"},
           "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                            "sample": sample}}
    print(json.dumps(rec), flush=True)


if __name__ == "__main__":
    main()

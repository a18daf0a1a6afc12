"""Benchmark of the paged-attention hot path on one GB300 (or N replicas).

Headline workload: the GQA decode batch with the Llama-3-8B attention shape
(64 requests x 1 query, seq_lens U[128, 4096], 32 q / 8 kv heads, head_size
128, block_size 16, bf16).  One step = the whole decode hot path on that
batch: the cache write of the step's 64 new tokens, split-KV stage 1 with the
page's split rule, and the LSE merge.  ``value`` is decode KV throughput in
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


def device_pool(shape, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


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
        self.S = pa.pa_num_kv_splits(self.max_seq, pa.pa_device_sm_count())
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
    """The oracle, as it stands, on a bounded sample of the decode batch:
    whole requests in order until ~budget_s of CPU work.  Returns
    (GB/s of KV processed, threads, sample description)."""
    import oracle
    threads = threads or (os.cpu_count() or 1)
    pool = oracle.reshape_and_cache(b.key, b.value, b.pool, b.slot_mapping, b.block_size)
    done_bytes, elapsed, n = 0, 0.0, 0
    per_tok = b.num_kv_heads * b.head_size * 2 * 2
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
        f"through the {b.num_seqs}-request GQA decode batch, {elapsed:.1f} s of {threads} threads")


# ---------------------------------------------------------------------------
# Secondary workloads (kernels timed alone, events on the launch stream).
# ---------------------------------------------------------------------------

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


def bench_prefill(pa, device, pk, flush, reps=10):
    """Chunked prefill: the varlen kernel on its own."""
    b = workloads.chunked_prefill(with_pool=False)
    pool = device_pool((b.num_blocks, 2, b.block_size, b.num_kv_heads, b.head_size), 3, device)
    q = to_dev_bf16(b.q, device)
    table, qsl = to_dev(b.block_table, torch.int32, device), to_dev(b.query_start_loc,
                                                                     torch.int32, device)
    seq = to_dev(b.seq_lens, torch.int32, device)
    out = torch.empty_like(q)
    lse = torch.empty((b.num_tokens, b.num_q_heads), dtype=torch.float32, device=device)
    mq = int(b.query_lens.max())

    def prefill():
        pa.pa_varlen_fwd(q, pool, table, qsl, seq, mq, b.scale, out=out, lse=lse)
    ms = _timed_with_flush(prefill, flush, reps)
    warm = time_events(prefill, reps)
    tf = b.causal_flops() / (ms * 1e-3) / 1e12
    res = {"workload": b.name, "kernel": "varlen_fwd", "ms": ms, "warm_ms": warm,
                              "tflops": tf, "causal_flops": b.causal_flops(),
                              "frac_of_bf16_peak": tf / pk["bf16_tflops"],
                              "peak": "bf16_tflops (measured burst)" if pk["source"] == "measured"
                              else "fallback"}
    del pool, q, out
    torch.cuda.empty_cache()
    return res


def bench_long_decode(pa, device, pk, flush, reps=10):
    """Long-context split-KV decode (8 x 131072)."""
    b = workloads.long_decode(with_pool=False)
    pool = device_pool((b.num_blocks, 2, b.block_size, b.num_kv_heads, b.head_size), 4, device)
    N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
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
    res = {"workload": b.name, "num_splits": S, "stage1_ms": st1, "stage1_warm_ms": warm,
                          "decode_plus_merge_ms": both, "kv_bytes": b.kv_bytes(),
                          "stage1_gbs": gbs, "frac_of_hbm_peak": gbs / pk["hbm_gbs"],
                          "step_gbs": b.kv_bytes() / (both * 1e-3) / 1e9,
                          "l2": "2 rotating pool copies"}
    del pool, pools, q, ws
    torch.cuda.empty_cache()
    return res


def bench_mla(pa, device, pk, flush, reps=10):
    """MLA latent decode (DeepSeek-V3 shape)."""
    m = workloads.mla_decode(with_pool=False)
    pool = device_pool((m.num_blocks, m.block_size, m.kv_lora_rank + m.rope_dim), 5, device)
    q = to_dev_bf16(m.q, device)
    table, seq = to_dev(m.block_table, torch.int32, device), to_dev(m.seq_lens, torch.int32,
                                                                    device)
    S = mla_splits(m, pa.pa_device_sm_count())
    ws = pa.decode_workspace(m.batch, m.num_heads, S, m.kv_lora_rank, device=device)
    o = torch.empty((m.batch, m.num_heads, m.kv_lora_rank), dtype=torch.bfloat16, device=device)
    lo = torch.empty((m.batch, m.num_heads), dtype=torch.float32, device=device)
    mx = int(m.seq_lens.max())
    pools = [pool, pool.clone()]
    mla = [lambda p=p: pa.pa_mla_decode(q, p, table, seq, m.scale, ws, o, lo, max_seq_len=mx)
           for p in pools]
    ms = _timed_rotating(mla, reps)
    warm = time_events(mla[0], reps)
    # The step's cache write of the 128 new latent rows, timed alone.
    kv_c, k_pe, slots = workloads.mla_new_tokens(m)
    d_kv_c, d_k_pe = to_dev_bf16(kv_c, device), to_dev_bf16(k_pe, device)
    d_slots = to_dev(slots, torch.int64, device)
    write_ms = _timed_with_flush(lambda: pa.pa_mla_cache_write(d_kv_c, d_k_pe, pool, d_slots),
                                 flush, reps)
    gbs = m.kv_bytes() / (ms * 1e-3) / 1e9
    flops = int(m.seq_lens.astype(np.int64).sum()) * m.num_heads * 2 * (
        m.kv_lora_rank + m.rope_dim + m.kv_lora_rank)
    res = {"workload": m.name, "num_splits": S, "ms": ms, "warm_ms": warm, "kv_bytes": m.kv_bytes(),
                         "gbs": gbs, "frac_of_hbm_peak": gbs / pk["hbm_gbs"],
                         "tflops": flops / (ms * 1e-3) / 1e12,
                         "cache_write_us": write_ms * 1e3, "cache_write_tokens": int(m.batch),
                         "l2": "2 rotating pool copies (cache write: L2 flushed)"}
    del pool, pools, q, ws
    torch.cuda.empty_cache()
    return res


def bench_mla_prefill(pa, device, pk, flush, reps=10):
    """MLA chunked prefill, multi-head formulation (DeepSeek-V3 shape): the
    kv_b_proj expansion of every context token and the attention over the
    expanded keys and values, timed together and apart."""
    m = workloads.mla_prefill(with_pool=False)
    pool = device_pool((m.num_blocks, m.block_size, m.kv_lora_rank + m.rope_dim), 7, device)
    q = to_dev_bf16(m.q, device)
    w = to_dev_bf16(m.w_kv_b, device)
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
    call = lambda: pa.pa_mla_prefill(q, pool, w, table, qsl, seq, mq, m.scale, ws, S, out=out,
                                     lse=lse)
    total = _timed_with_flush(call, flush, reps)
    warm = time_events(call, reps)
    expand = _timed_with_flush(lambda: pa.pa_mla_expand_kv(pool, w, table, seq, k_ws, v_ws),
                               flush, reps)
    attn = total - expand
    ef, af = m.expand_flops(), m.causal_flops()
    res = {"workload": m.name, "ms": total, "warm_ms": warm, "expand_ms": expand,
           "attention_ms": attn,
           "expand_tflops": ef / (expand * 1e-3) / 1e12,
           "attention_tflops": af / (attn * 1e-3) / 1e12,
           "tflops": (ef + af) / (total * 1e-3) / 1e12,
           "frac_of_bf16_peak": (ef + af) / (total * 1e-3) / 1e12 / pk["bf16_tflops"],
           "expanded_bytes": kv_elems * 320 * 2}
    del pool, q, w, ws
    torch.cuda.empty_cache()
    return res


def device_fp8_pool(shape, seed, device):
    """Uniformly random finite e4m3 codes (the NaN codes 0x7F / 0xFF excluded),
    drawn on the device."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    r = torch.randint(0, 254, shape, generator=g, device=device, dtype=torch.uint8)
    r += (r >= 0x7F).to(torch.uint8)
    return r


def fp8_kernel_name(d, grp):
    """The fp8 stage-1 instantiation the library launches: groups of more
    than 8 heads take two n-tiles (and, for d = 128, a fourth ring stage)."""
    wide = grp > 8
    stages = (4 if wide else 3) if d == 128 else 8
    return f"decode_splitkv_fp8_kernel<{d},{stages},{2 if wide else 1}>"


def bench_fp8_decode(pa, device, pk, flush, reps=10):
    """Split-KV decode over an fp8 (e4m3) pool, on the GQA decode batch and the
    long-context batch: stage 1 alone, and the whole step (quantising cache
    write + stage 1 + merge)."""
    res = {}
    ks, vs = workloads.FP8_K_SCALE, workloads.FP8_V_SCALE
    for make, seed in ((workloads.gqa_decode, 12), (workloads.long_decode, 14)):
        b = make(with_pool=False)
        N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
        pool = device_fp8_pool((b.num_blocks, 2, b.block_size, b.num_kv_heads, d), seed, device)
        q = to_dev_bf16(b.q, device).view(N, hq, d)
        key, value = to_dev_bf16(b.key, device), to_dev_bf16(b.value, device)
        slots = to_dev(b.slot_mapping, torch.int64, device)
        table = to_dev(b.block_table, torch.int32, device)
        seq = to_dev(b.seq_lens, torch.int32, device)
        mx = int(b.seq_lens.max())
        S = pa.pa_num_kv_splits(mx, pa.pa_device_sm_count())
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
        res[b.name] = {"num_splits": S, "stage1_ms": st1, "stage1_warm_ms": warm,
                       "step_ms": both, "kv_bytes": kv,
                       "stage1_gbs": gbs, "frac_of_hbm_peak": gbs / pk["hbm_gbs"],
                       "step_gbs": kv / (both * 1e-3) / 1e9,
                       "kernel": fp8_kernel_name(d, b.num_q_heads // b.num_kv_heads),
                       "l2": "2 rotating pool copies"}
        del pool, pools, q, ws
        torch.cuda.empty_cache()
    return res


def bench_cascade(pa, device, pk, flush, reps=10):
    """Cascade attention on 64 decode requests sharing a prompt (4096 tokens:
    17 MB of K/V per layer, L2-resident; 32768 tokens: 134 MB, more than L2),
    against plain split-KV decode of the same batch, which reads the prompt
    once per request."""
    res = {}
    for prefix in (4096, 32768):
        b = workloads.shared_prefix_decode(prefix_tokens=prefix, with_pool=False)
        N, hq, d = b.num_seqs, b.num_q_heads, b.head_size
        pool = device_pool((b.num_blocks, 2, b.block_size, b.num_kv_heads, d), 6, device)
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
        casc = _timed_with_flush(lambda: pa.pa_cascade_fwd(q, pool, table, qsl, seq, 1, P, b.scale,
                                                           cws, S1, mx, out=o, lse=lo),
                                 flush, reps)
        row = b.num_kv_heads * d * 2 * 2
        unique = (prefix + int((b.seq_lens - prefix).astype(np.int64).sum())) * row
        res[b.name] = {"prefix_tokens": prefix, "prefix_splits": S1, "suffix_splits": S2,
                       "cascade_ms": casc, "plain_decode_ms": plain, "speedup": plain / casc,
                       "unique_kv_bytes": unique,
                       "cascade_unique_gbs": unique / (casc * 1e-3) / 1e9,
                       "plain_kv_bytes": b.kv_bytes()}
        del pool, q, ws, cws
        torch.cuda.empty_cache()
    return res


SECONDARY = {"chunked_prefill": bench_prefill, "long_decode": bench_long_decode,
             "mla_decode": bench_mla, "fp8_decode": bench_fp8_decode, "cascade": bench_cascade,
             "mla_prefill": bench_mla_prefill}


def secondary(pa, device, pk):
    flush = l2_flusher(device)
    return {name: fn(pa, device, pk, flush) for name, fn in SECONDARY.items()}


def mla_splits(m, sms):
    """Splits for the MLA workload: each (request, split, 128-head group) runs
    on a pair of SMs, so enough splits to give every pair slot one unit, and
    no more (each split adds a 128 x 513 fp32 partial per request)."""
    groups = max(1, (m.num_heads + 127) // 128)
    return max(1, min(8, math.ceil((sms // 2) / (m.batch * groups))))


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
        rec = SECONDARY[args.only](pa, device, pk, l2_flusher(device), reps=args.steps)
        if rank == 0:
            print(json.dumps({"only": args.only, **rec}), flush=True)
        return

    b = workloads.gqa_decode()
    step = DecodeStep(pa, b, device)
    kv_bytes = b.kv_bytes()

    clocks = ClockSampler(local)
    clocks.start()
    for k in range(warmup):
        step.run(k)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record()
    for k in range(args.steps):
        step.run(k)
    t_end.record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    total_ms = t_start.elapsed_time(t_end)
    # The stage-1 kernel's own duration, from a second pass over the same K
    # steps with events on its stream around every stage-1 launch.  Events
    # between the step's kernels serialise their programmatic dependent
    # launches (about 8 us per step), so they stay out of the pass above.
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    for k in range(args.steps):
        step.run(k, ev[k])
    torch.cuda.synchronize()
    clk = clocks.stop()
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

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, sample = cpu_baseline_sample(b)
        cpu = {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}

    if rank == 0:
        rec = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded numpy N(0,1) rounded to bf16; random block permutation)",
            "config": {"workload": b.name, "num_seqs": b.num_seqs, "seq_lens": "U[128,4096]",
                       "num_q_heads": 32, "num_kv_heads": 8, "head_size": 128,
                       "block_size": 16, "num_splits": step.S, "kv_bytes_per_step": kv_bytes,
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

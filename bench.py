#!/usr/bin/env python
"""Throughput of the rotated, block-quantized KV-cache hot path on GB300.

A step = one decode step of the 64k-context workload (4 sequences x 65,536
tokens, 24 query / 4 KV heads, head_dim 256, K q8_0 / V q4_0, bf16 tail of
1024 tokens): rotate + quantize + append one new token per sequence, then
decode attention over body + tail for all 24 heads.  The value is achieved
HBM bandwidth in GB/s: algorithmic bytes (packed body + bf16 tail + q/out of
the decode, plus the append's input, packed output and tail writes) divided by
the measured step time.  Inputs are larger than L2 (446 MB per step), so no
flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torch.distributed.run: every rank holds its own replica of
the workload (the path shards over (sequence, KV head) with no exchange), and
the value is the bytes of all ranks over the slowest rank's time.
--impl reference times the CPU oracle (numpy, float64) on a bounded sample of
the same workload on the host cores; it is test infrastructure, not a product
path.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rotated_bit_kv_kvq_gb300 import workloads as wl  # noqa: E402

METRIC = "quantized-KV decode attention: achieved HBM GB/s vs 8 TB/s; append tokens/s"
BLOCK_BYTES = {"q4_0": 18, "q5_0": 22, "q8_0": 34, "q4_1": 20, "q5_1": 24}


# ---------------------------------------------------------------------------
# byte accounting (algorithmic bytes)
# ---------------------------------------------------------------------------
def token_bytes(w: wl.Workload) -> int:
    """Packed body bytes of one token of one KV head, K + V."""
    nb = w.head_dim // 32
    return nb * (BLOCK_BYTES[w.k_type] + BLOCK_BYTES[w.v_type])


def decode_bytes(w: wl.Workload, lengths, q_bytes=2, out_bytes=2) -> int:
    tot = 0
    for n in lengths:
        body = max(0, int(n) - w.tail_len)
        tail = min(int(n), w.tail_len)
        tot += w.n_kv_heads * (body * token_bytes(w) + tail * 2 * w.head_dim * 2)
    tot += len(lengths) * w.n_q_heads * w.head_dim * (q_bytes + out_bytes)
    return tot


def append_bytes(w: wl.Workload, n_new: int, in_bytes=2) -> int:
    """Input K+V read, packed blocks written, and bf16 tail rows written (only the
    last min(n_new, tail_len) tokens of a call reach the ring)."""
    heads = w.n_kv_heads * w.batch
    tail_tokens = min(n_new, w.tail_len)
    return heads * (n_new * (2 * w.head_dim * in_bytes + token_bytes(w)) + tail_tokens * 2 * w.head_dim * 2)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def recorded_traffic(kernel_file: str):
    """ncu DRAM bytes per launch recorded in profiles/, valid only while the
    kernel source is unchanged (its hash is stored beside the number)."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "decode_b4_ctx64k_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    src = os.path.join(ROOT, "rotated_bit_kv_kvq_gb300", "csrc", kernel_file)
    h = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return d.get("bytes_per_launch") if d.get("source_sha256") == h else None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,utilization.gpu")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        self.path = os.path.join("/tmp", f"kvq_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, loaded, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                clk, cmax = float(parts[1]), float(parts[2])
            except ValueError:
                continue
            sm.append(clk)
            mx.append(cmax)
            try:
                util = float(parts[9]) if len(parts) > 9 else None
            except ValueError:
                util = None
            if util is not None and util >= 50.0:  # a sample taken while the GPU ran our kernels
                loaded.append(clk)
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        pick = loaded if loaded else sm
        return {"sm_mhz": statistics.median(pick) if pick else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(loaded)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def fill_cache(torch, kvq, cache, w: wl.Workload, n_fill: int, seed: int = 0):
    """Seeded synthetic history (N(0,1), outlier channels x20, bf16), appended
    through the library's own write path in chunks."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k_chan = wl.outlier_channels(rng, w.n_kv_heads, w.head_dim, w.n_outliers)
    v_chan = wl.outlier_channels(rng, w.n_kv_heads, w.head_dim, w.n_outliers)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    kmask = torch.ones(w.n_kv_heads, w.head_dim, device="cuda")
    vmask = torch.ones(w.n_kv_heads, w.head_dim, device="cuda")
    for h in range(w.n_kv_heads):
        kmask[h, torch.tensor(k_chan[h])] = 20.0
        vmask[h, torch.tensor(v_chan[h])] = 20.0
    chunk = 8192
    done = 0
    while done < n_fill:
        n = min(chunk, n_fill - done)
        k = (torch.randn(w.batch, n, w.n_kv_heads, w.head_dim, generator=gen, device="cuda") * kmask).to(torch.bfloat16)
        v = (torch.randn(w.batch, n, w.n_kv_heads, w.head_dim, generator=gen, device="cuda") * vmask).to(torch.bfloat16)
        kvq.kvq_rotate_quantize_append(cache.desc, k, v)
        done += n
    torch.cuda.synchronize()
    st, bits = kvq.kvq_sync_status(cache.desc)
    assert st == 0, (st, bits)
    return kmask, vmask, gen


def max_over_ranks(vals, world: int, device: str = "cpu"):
    """Every rank calls this with its own timings; each comes back as the maximum
    over the ranks (the slowest replica sets the job's time)."""
    import torch
    t = torch.tensor(vals, dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_gbs(world: int, bytes_per_rank_step: float, ms_per_step: float) -> float:
    """Whole-job throughput: every rank moves the same bytes per step (weak scaling,
    one replica per GPU), over the slowest rank's step time."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def hold_device(torch, cycles: int = 200_000):
    """Keep the GPU busy for ~0.1 ms (a device-side wait on the current stream) while
    the host enqueues the first calls of a timed region: the start event then fires
    with those calls already queued, so the region between the events holds their
    device work and not the host's launch latency of the first call."""
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        sleep(cycles)


def run_ours(args):
    import torch
    import torch.distributed as dist

    from rotated_bit_kv_kvq_gb300 import kvq

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    w = wl.WORKLOADS[args.workload]
    if args.ctx:
        w = w.scaled(ctx=args.ctx)
    K, W = args.steps, args.warmup
    n_new = max(1, w.append_per_step)
    extra = (W + K) * n_new
    n_start = w.ctx - n_new                       # first timed step decodes at exactly ctx tokens
    n_fill = n_start - W * n_new
    cache = kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, w.max_ctx(extra + 64), w.tail_len, w.k_type, w.v_type)
    kmask, vmask, gen = fill_cache(torch, kvq, cache, w, n_fill, seed=rank)

    # per-step inputs, generated ahead of the timed region
    P = 8
    ks = [(torch.randn(w.batch, n_new, w.n_kv_heads, w.head_dim, generator=gen, device="cuda") * kmask).to(torch.bfloat16)
          for _ in range(P)]
    vs = [(torch.randn(w.batch, n_new, w.n_kv_heads, w.head_dim, generator=gen, device="cuda") * vmask).to(torch.bfloat16)
          for _ in range(P)]
    qs = [torch.randn(w.batch, w.n_q_heads, w.head_dim, generator=gen, device="cuda").to(torch.bfloat16) for _ in range(P)]
    out = torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(kvq.kvq_decode_workspace_bytes(cache.desc, w.n_q_heads), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    seq0 = cache.seq_len.clone()

    # one step = kvq_append_decode: the new token is written inside the decode launch
    # (split + merge kernels) when the workload allows it (tail present, <= 8 query heads
    # per KV head, one tail split), else append + decode
    fused = w.tail_len > 0 and n_new <= w.tail_len and w.group <= 8 and w.tail_len <= 4096
    launches_per_step = 2 if fused else 3

    def step(i):
        kvq.kvq_append_decode(cache.desc, ks[i % P], vs[i % P], qs[i % P], out, ws, stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()

    # ---- device-resident timed region: W warm-up steps, then K steps --------------
    for i in range(W):
        step(i)
    torch.cuda.synchronize()
    lens_first = cache.seq_len.cpu().numpy() + n_new
    clocks = ClockSampler(local)
    clocks.start()
    # the sampler's first 0.3 s: decode calls (reads only; the cache is not advanced),
    # so that the timed region starts on a GPU at its working clocks, not one coming
    # out of an idle pause
    t_pre = time.perf_counter()
    n_pre = 0
    while time.perf_counter() - t_pre < 0.3:
        for _ in range(50):
            kvq.kvq_decode_attention(cache.desc, qs[n_pre % P], out, ws, stream=stream)
            n_pre += 1
        torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_device(torch)
    e0.record(stream)
    for i in range(K):
        step(W + i)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    step_ms = e0.elapsed_time(e1) / K
    # keep the GPU under the same decode load for a while longer, so that the clock
    # samples (every 100 ms) are taken under load; the metric is not timed here
    t_load = time.perf_counter()
    n_load = 0
    while time.perf_counter() - t_load < args.load_s:
        for _ in range(50):
            kvq.kvq_decode_attention(cache.desc, qs[n_load % P], out, ws, stream=stream)
            n_load += 1
        torch.cuda.synchronize()
    clk = clocks.stop()
    clk["load_s"] = round(time.perf_counter() - t_load, 2)
    clk["load_calls"] = n_load
    st, bits = kvq.kvq_sync_status(cache.desc)
    assert st == 0, (st, bits)
    total_bytes = 0
    for i in range(K):
        lens = lens_first + i * n_new
        total_bytes += decode_bytes(w, lens) + append_bytes(w, n_new)

    # ---- decode kernel alone (the dominant kernel), same context --------------------
    dec_lens = cache.seq_len.cpu().numpy()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(3):
        kvq.kvq_decode_attention(cache.desc, qs[i % P], out, ws, stream=stream)
    torch.cuda.synchronize()
    hold_device(torch)
    d0.record(stream)
    for i in range(K):
        kvq.kvq_decode_attention(cache.desc, qs[i % P], out, ws, stream=stream)
    d1.record(stream)
    torch.cuda.synchronize()
    dec_ms = d0.elapsed_time(d1) / K
    dec_bytes = decode_bytes(w, dec_lens)
    # the same calls timed one by one (an event pair around each) for the spread
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for i in range(K):
        evs[i][0].record(stream)
        kvq.kvq_decode_attention(cache.desc, qs[i % P], out, ws, stream=stream)
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    dec_each = sorted(a.elapsed_time(b) for a, b in evs)
    dec_spread = {"median": round(statistics.median(dec_each), 5),
                  "p10": round(dec_each[int(0.1 * (K - 1))], 5), "p90": round(dec_each[int(0.9 * (K - 1))], 5),
                  "n": K}

    # ---- append alone (one token per sequence) ----------------------------------------
    cache.seq_len.copy_(seq0)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a0.record(stream)
    for i in range(K):
        kvq.kvq_rotate_quantize_append(cache.desc, ks[i % P], vs[i % P], stream=stream)
    a1.record(stream)
    torch.cuda.synchronize()
    app_eager_ms = a0.elapsed_time(a1) / K
    # the same K calls captured in one CUDA graph: the calls' device time without
    # the host's per-launch cost (a one-token append is a few microseconds of work)
    cap_a = torch.cuda.Stream()
    g_app = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_app, stream=cap_a):
        for i in range(K):
            kvq.kvq_rotate_quantize_append(cache.desc, ks[i % P], vs[i % P], stream=cap_a)
    cache.seq_len.copy_(seq0)
    torch.cuda.synchronize()
    with torch.cuda.stream(cap_a):
        a0.record(cap_a)
        g_app.replay()
        a1.record(cap_a)
    torch.cuda.synchronize()
    app_ms = a0.elapsed_time(a1) / K
    del g_app

    # ---- end to end through the public API, host buffers -----------------------------
    # Every step copies the new tokens and the query from pinned host memory, runs
    # kvq_append_decode and reads the output back to the host.  The step's inputs sit
    # in one pinned buffer per slot ([k | v | q], 16-byte aligned parts), so one copy
    # moves them; the call gets views of the device copy.  "e2e" replays that step
    # captured in a CUDA graph (one per input slot: the serving form); "e2e_eager"
    # issues the same calls one by one.
    parts = [ks[0], vs[0], qs[0]]
    nbytes_in = [t.numel() * t.element_size() for t in parts]
    offs = [0, nbytes_in[0], nbytes_in[0] + nbytes_in[1]]
    assert all(o % 16 == 0 for o in offs)
    hin = []
    for slot in range(P):
        hb = torch.empty(sum(nbytes_in), dtype=torch.uint8).pin_memory()
        for t, o, nb in zip((ks[slot], vs[slot], qs[slot]), offs, nbytes_in):
            hb[o:o + nb].copy_(t.contiguous().view(torch.uint8).reshape(-1).cpu())
        hin.append(hb)
    din = torch.empty(sum(nbytes_in), dtype=torch.uint8, device="cuda")
    dk, dv, dq = [din[o:o + nb].view(t.dtype).view(t.shape) for t, o, nb in zip(parts, offs, nbytes_in)]
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_body(i, s):
        din.copy_(hin[i % P], non_blocking=True)
        kvq.kvq_append_decode(cache.desc, dk, dv, dq, out, ws, stream=s)
        hout.copy_(out, non_blocking=True)

    def timed_loop(run_step):
        cache.seq_len.copy_(seq0)
        torch.cuda.synchronize()
        for i in range(W):
            run_step(i)
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(K):
            run_step(W + i)
        t1 = time.perf_counter()
        barrier()
        return (t1 - t0) * 1e3 / K

    def eager_step(i):
        e2e_body(i, stream)
        stream.synchronize()

    e2e_eager_ms = timed_loop(eager_step)
    cap = torch.cuda.Stream()
    graphs = []
    for slot in range(P):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            e2e_body(slot, cap)
        graphs.append(g)

    def graph_step(i):
        graphs[i % P].replay()
        torch.cuda.current_stream().synchronize()

    e2e_ms = timed_loop(graph_step)
    st, bits = kvq.kvq_sync_status(cache.desc)
    assert st == 0, (st, bits)
    h2d = sum(t.numel() * t.element_size() for t in (ks[0], vs[0], qs[0]))
    d2h = out.numel() * out.element_size()

    # ---- max over ranks -----------------------------------------------------------------
    step_ms, dec_ms, app_ms, app_eager_ms, e2e_ms, e2e_eager_ms = max_over_ranks(
        [step_ms, dec_ms, app_ms, app_eager_ms, e2e_ms, e2e_eager_ms], world, "cuda")

    if rank == 0:
        peak, peak_kind = measured_peaks()
        achieved = dec_bytes / (dec_ms * 1e-3) / 1e9
        per_step_bytes = total_bytes / K
        line = {
            "metric": METRIC,
            "value": round(job_gbs(world, per_step_bytes, step_ms), 2),
            "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": round(step_ms, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "q8_0/q4_0 codes -> fp16 mma, fp32 accumulate",
            "data": "synthetic (seeded N(0,1), 4 outlier channels x20 per KV head, bf16)",
            "config": {"workload": w.name, "batch": w.batch, "ctx": w.ctx, "q_heads": w.n_q_heads,
                       "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "k_type": w.k_type, "v_type": w.v_type,
                       "tail_len": w.tail_len, "append_per_step": n_new,
                       "l2": config_l2_note(w),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": "decode (split-K + combine) at ctx "
                         f"{int(dec_lens.max())}", "achieved": round(achieved, 1), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "bytes_per_launch": int(dec_bytes), "ms_per_launch": round(dec_ms, 5),
                         "traffic": recorded_traffic("kvq_decode_impl.cuh"),
                         "ms_per_launch_each": dec_spread},
            "append": {"tokens_per_s": round(world * w.batch * n_new / (app_ms * 1e-3), 1),
                       "ms_per_call": round(app_ms, 5), "ms_per_call_eager": round(app_eager_ms, 5),
                       "how": "kvq_rotate_quantize_append, one token per sequence, K calls in one CUDA graph "
                              "(device time); ms_per_call_eager: the same calls launched one by one"},
            "e2e": {"value": round(job_gbs(world, per_step_bytes, e2e_ms), 2), "unit": "GB/s",
                    "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "how": "CUDA graph per step: one pinned H2D copy of the step's k, v, q + kvq_append_decode "
                           "+ D2H of the output, host sync each step"},
            "e2e_eager": {"value": round(job_gbs(world, per_step_bytes, e2e_eager_ms), 2), "unit": "GB/s",
                          "ms_per_step": round(e2e_eager_ms, 5)},
            "gpu_launches": launches_per_step * K,
            "step_call": "kvq_append_decode" + (" (append fused into the decode launch)" if fused else ""),
            "clocks": clk,
        }
        if not args.no_configs:
            line["configs"] = run_config_legs(torch, kvq, peak)
        if not args.no_prefill:
            line["prefill"] = run_prefill_bench(torch, kvq, max(5, K // 5), 3)
        if not args.no_format_pairs:
            del cache, ws
            torch.cuda.empty_cache()
            line["format_pairs"] = run_format_pairs(torch, kvq, w, max(5, K // 5), peak)
            line["paged"] = run_format_pairs(torch, kvq, w, max(5, K // 5), peak,
                                             pairs=((w.k_type, w.v_type),), page_tokens=256)[0]
            line["outliers"] = run_format_pairs(torch, kvq, w, max(5, K // 5), peak,
                                                pairs=((w.k_type, w.v_type),), outliers=True)[0]
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w, budget_s=args.cpu_budget)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def config_l2_note(w: wl.Workload) -> str:
    """How the timed region keeps the cache out of L2 (same words for both arms)."""
    return "inputs larger than L2 (446 MB per step), no flush" if w.name == wl.HEADLINE else \
        "L2 flushed (256 MB written) before each timed call when the call's bytes fit in L2"


# ---------------------------------------------------------------------------
# the other decode workloads: decode call alone, per-call device time
# ---------------------------------------------------------------------------
CONFIG_LEGS = ("decode_d64_ctx256", "decode_gqa16x8_ctx4k", "decode_b32_ragged8k")


def fill_cache_ragged(torch, kvq, cache, w: wl.Workload, lens, seed: int = 0):
    """Seeded synthetic history (as fill_cache) appended to each sequence up to its own
    length, through the library's write path (per-sequence counts)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k_chan = wl.outlier_channels(rng, w.n_kv_heads, w.head_dim, w.n_outliers)
    v_chan = wl.outlier_channels(rng, w.n_kv_heads, w.head_dim, w.n_outliers)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    kmask = torch.ones(w.n_kv_heads, w.head_dim, device="cuda")
    vmask = torch.ones(w.n_kv_heads, w.head_dim, device="cuda")
    for h in range(w.n_kv_heads):
        kmask[h, torch.tensor(k_chan[h])] = 20.0
        vmask[h, torch.tensor(v_chan[h])] = 20.0
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    lens = np.asarray(lens, dtype=np.int64)
    chunk, done = 8192, 0
    while done < int(lens.max()):
        n = min(chunk, int(lens.max()) - done)
        per = torch.tensor(np.clip(lens - done, 0, n), dtype=torch.int32, device="cuda")
        k = (torch.randn(w.batch, n, w.n_kv_heads, w.head_dim, generator=gen, device="cuda") * kmask).to(dt)
        v = (torch.randn(w.batch, n, w.n_kv_heads, w.head_dim, generator=gen, device="cuda") * vmask).to(dt)
        kvq.kvq_rotate_quantize_append(cache.desc, k, v, n_new_per_seq=per)
        done += n
    torch.cuda.synchronize()
    st, bits = kvq.kvq_sync_status(cache.desc)
    assert st == 0, (st, bits)
    assert np.array_equal(cache.seq_len.cpu().numpy(), lens)
    return gen


def run_config_legs(torch, kvq, peak: float, iters: int = 40):
    """The decode call alone on the other workloads, each at its own shapes, formats,
    dtypes and (ragged) lengths.  Calls whose bytes fit in L2 are timed one by one with
    L2 flushed (a 256 MB buffer written) before each; larger ones back to back."""
    res = []
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for name in CONFIG_LEGS:
        w = wl.WORKLOADS[name]
        rng = np.random.Generator(np.random.PCG64(0))
        if w.ragged_min is not None:
            lens = rng.integers(w.ragged_min, w.ctx + 1, size=w.batch).astype(np.int64)
        else:
            lens = np.full(w.batch, w.ctx, dtype=np.int64)
        cache = kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, w.max_ctx(64), w.tail_len, w.k_type, w.v_type)
        gen = fill_cache_ragged(torch, kvq, cache, w, lens)
        dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        qs = [torch.randn(w.batch, w.n_q_heads, w.head_dim, generator=gen, device="cuda").to(dt) for _ in range(4)]
        out = torch.empty(w.batch, w.n_q_heads, w.head_dim, dtype=dt, device="cuda")
        ws = torch.empty(kvq.kvq_decode_workspace_bytes(cache.desc, w.n_q_heads), dtype=torch.uint8, device="cuda")
        esz = 2 if w.dtype == "bf16" else 4
        nbytes = decode_bytes(w, lens, q_bytes=esz, out_bytes=esz)
        fits = nbytes < 100e6
        for i in range(3):
            kvq.kvq_decode_attention(cache.desc, qs[i % 4], out, ws, stream=stream)
        torch.cuda.synchronize()
        times = []
        if fits:
            for i in range(iters):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                kvq.kvq_decode_attention(cache.desc, qs[i % 4], out, ws, stream=stream)
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = statistics.median(times)
        else:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(iters):
                kvq.kvq_decode_attention(cache.desc, qs[i % 4], out, ws, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / iters
        st, bits = kvq.kvq_sync_status(cache.desc)
        assert st == 0, (st, bits)
        gbs = nbytes / (ms * 1e-3) / 1e9
        res.append({"workload": name, "batch": w.batch, "ctx": w.ctx,
                    "lengths": "uniform %d..%d (seed 0), total %d" % (w.ragged_min, w.ctx, int(lens.sum()))
                    if w.ragged_min is not None else "all %d" % w.ctx,
                    "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads, "head_dim": w.head_dim,
                    "k_type": w.k_type, "v_type": w.v_type, "tail_len": w.tail_len, "q_dtype": w.dtype,
                    "ms_per_call": round(ms, 5), "bytes_per_call": int(nbytes), "gbs": round(gbs, 1),
                    "frac": round(gbs / peak, 4),
                    "l2": "flushed before each call (bytes fit in L2)" if fits else "larger than L2, back to back"})
        del cache, ws, qs, out
        torch.cuda.empty_cache()
    del flush
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# the same decode workload with the scale + minimum formats in the K/V pairs the
# benchmark summary names (q5_0-q4_1, q8_0-q5_1): decode call alone, same context
# ---------------------------------------------------------------------------
FORMAT_PAIRS = (("q5_0", "q4_1"), ("q8_0", "q5_1"))


def outlier_lists(w: wl.Workload, seed: int) -> np.ndarray:
    """Per KV head, 32 channels kept at 8 bits: the synthetic history's K and V
    outlier channels (the draws fill_cache makes with the same seed), then the
    lowest other channels, sorted."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k_chan = wl.outlier_channels(rng, w.n_kv_heads, w.head_dim, w.n_outliers)
    v_chan = wl.outlier_channels(rng, w.n_kv_heads, w.head_dim, w.n_outliers)
    out = []
    for h in range(w.n_kv_heads):
        chosen = sorted(set(k_chan[h].tolist()) | set(v_chan[h].tolist()))[:32]
        rest = [c for c in range(w.head_dim) if c not in chosen]
        out.append(sorted(chosen + rest[:32 - len(chosen)]))
    return np.asarray(out, dtype=np.int64)


def run_format_pairs(torch, kvq, w: wl.Workload, steps: int, peak: float, pairs=FORMAT_PAIRS, page_tokens=0,
                     outliers=False):
    """Decode call alone at the workload's context for other K/V format pairs, or
    (page_tokens > 0) from a paged cache whose pages are handed out in a shuffled
    order (a pool with 5% spare pages), or (outliers) with 32 channels per KV head
    kept as unrotated q8_0 (their codes and scales add 2 x 34 bytes per body token
    and KV head)."""
    import dataclasses
    res = []
    for kt, vt in pairs:
        w2 = dataclasses.replace(w, k_type=kt, v_type=vt)
        max_ctx = w2.max_ctx(64)
        paged = {}
        if page_tokens:
            max_ctx = (max_ctx + page_tokens - 1) // page_tokens * page_tokens
            per_seq = max_ctx // page_tokens
            n_pages = w2.batch * per_seq + max(1, w2.batch * per_seq // 20)
            g = torch.Generator()
            g.manual_seed(5)
            table = torch.randperm(n_pages, generator=g)[:w2.batch * per_seq].to(torch.int32)
            paged = dict(page_tokens=page_tokens, n_pages=n_pages, page_table=table)
        extra = dict(outliers=outlier_lists(w2, 7).tolist()) if outliers else {}
        cache = kvq.KVCache(w2.batch, w2.n_kv_heads, w2.head_dim, max_ctx, w2.tail_len, kt, vt, **paged, **extra)
        _, _, gen = fill_cache(torch, kvq, cache, w2, w2.ctx, seed=7)
        qs = [torch.randn(w2.batch, w2.n_q_heads, w2.head_dim, generator=gen, device="cuda").to(torch.bfloat16)
              for _ in range(4)]
        out = torch.empty(w2.batch, w2.n_q_heads, w2.head_dim, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(kvq.kvq_decode_workspace_bytes(cache.desc, w2.n_q_heads), dtype=torch.uint8, device="cuda")
        stream = torch.cuda.current_stream()
        for i in range(3):
            kvq.kvq_decode_attention(cache.desc, qs[i % 4], out, ws, stream=stream)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        hold_device(torch)
        e0.record(stream)
        for i in range(steps):
            kvq.kvq_decode_attention(cache.desc, qs[i % 4], out, ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        st, bits = kvq.kvq_sync_status(cache.desc)
        assert st == 0, (st, bits)
        ms = e0.elapsed_time(e1) / steps
        lens = cache.seq_len.cpu().numpy()
        nbytes = decode_bytes(w2, lens)
        if outliers:
            nbytes += sum(max(0, int(n) - w2.tail_len) for n in lens) * w2.n_kv_heads * 2 * 34
        gbs = nbytes / (ms * 1e-3) / 1e9
        r = {"k_type": kt, "v_type": vt, "ctx": w2.ctx, "ms_per_call": round(ms, 5),
             "bytes_per_call": int(nbytes), "gbs": round(gbs, 1), "frac": round(gbs / peak, 4)}
        if page_tokens:
            r["page_tokens"] = page_tokens
            r["layout"] = "paged, shuffled page table"
        if outliers:
            r["n_outlier"] = 32
            # the write path of this cache: one 8,192-token append of the workload's sequences and heads
            kb = (torch.randn(w2.batch, 8192, w2.n_kv_heads, w2.head_dim, generator=gen, device="cuda")).to(torch.bfloat16)
            cache.seq_len.zero_()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            kvq.kvq_rotate_quantize_append(cache.desc, kb, kb, stream=stream)
            cache.seq_len.zero_()
            a0.record(stream)
            kvq.kvq_rotate_quantize_append(cache.desc, kb, kb, stream=stream)
            a1.record(stream)
            torch.cuda.synchronize()
            r["append_8192_ms"] = round(a0.elapsed_time(a1), 4)
        res.append(r)
        del cache, ws
        torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# prompt workload: bulk append of the prompt + causal prefill attention
# ---------------------------------------------------------------------------
def prefill_flops(w: wl.Workload) -> float:
    """Useful flops of causal attention: 4 * head_dim per visible (query, key) pair."""
    n = w.ctx
    return 4.0 * w.head_dim * (n * (n + 1) / 2) * w.n_q_heads * w.batch


def run_prefill_bench(torch, kvq, steps: int, warmup: int, seed: int = 0):
    w = wl.WORKLOADS["prefill_b2_4k"]
    cache = kvq.KVCache(w.batch, w.n_kv_heads, w.head_dim, w.max_ctx(), w.tail_len, w.k_type, w.v_type)
    rng = np.random.Generator(np.random.PCG64(seed))
    k_chan = wl.outlier_channels(rng, w.n_kv_heads, w.head_dim, w.n_outliers)
    v_chan = wl.outlier_channels(rng, w.n_kv_heads, w.head_dim, w.n_outliers)
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed + 1)
    kmask = torch.ones(w.n_kv_heads, w.head_dim, device="cuda")
    vmask = torch.ones(w.n_kv_heads, w.head_dim, device="cuda")
    for h in range(w.n_kv_heads):
        kmask[h, torch.tensor(k_chan[h])] = 20.0
        vmask[h, torch.tensor(v_chan[h])] = 20.0
    shape = (w.batch, w.ctx, w.n_kv_heads, w.head_dim)
    k = (torch.randn(shape, generator=gen, device="cuda") * kmask).to(torch.bfloat16)
    v = (torch.randn(shape, generator=gen, device="cuda") * vmask).to(torch.bfloat16)
    q = torch.randn((w.batch, w.ctx, w.n_q_heads, w.head_dim), generator=gen, device="cuda").to(torch.bfloat16)
    out = torch.empty_like(q)
    ws = torch.empty(kvq.kvq_prefill_workspace_bytes(cache.desc, w.n_q_heads, w.ctx), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.current_stream()
    # append: the whole prompt of both sequences per call, into an emptied cache
    app = []
    for i in range(warmup + steps):
        cache.seq_len.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        kvq.kvq_rotate_quantize_append(cache.desc, k, v, stream=stream)
        e1.record(stream)
        app.append((e0, e1))
    torch.cuda.synchronize()
    app_ms = statistics.median(a.elapsed_time(b) for a, b in app[warmup:])
    for i in range(warmup):
        kvq.kvq_prefill_attention(cache.desc, q, out, ws, chunk=w.chunk, stream=stream)
    torch.cuda.synchronize()
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    hold_device(torch)
    p0.record(stream)
    for i in range(steps):
        kvq.kvq_prefill_attention(cache.desc, q, out, ws, chunk=w.chunk, stream=stream)
    p1.record(stream)
    torch.cuda.synchronize()
    st, bits = kvq.kvq_sync_status(cache.desc)
    assert st == 0, (st, bits)
    att_ms = p0.elapsed_time(p1) / steps
    tokens = w.batch * w.ctx
    app_bytes = append_bytes(w, w.ctx)
    flops = prefill_flops(w)
    peak = None
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peak = float(json.load(open(pk))["bf16_tflops"])
    tflops = flops / (att_ms * 1e-3) / 1e12
    return {"workload": w.name, "batch": w.batch, "prompt": w.ctx, "q_heads": w.n_q_heads,
            "kv_heads": w.n_kv_heads, "head_dim": w.head_dim, "k_type": w.k_type, "v_type": w.v_type,
            "tail_len": w.tail_len, "causal": True,
            "append": {"ms_per_call": round(app_ms, 4), "tokens_per_s": round(tokens / (app_ms * 1e-3), 1),
                       "gbs": round(app_bytes / (app_ms * 1e-3) / 1e9, 1)},
            "attention": {"ms_per_call": round(att_ms, 4), "useful_flops": flops,
                          "tflops": round(tflops, 1), "bound": "tensor", "peak_tflops": peak,
                          "peak_kind": "measured bf16 burst (the fp16 dense rate is the same)" if peak else None,
                          "frac": round(tflops / peak, 4) if peak else None,
                          "note": "fp16 UMMA, three products per contraction (hi/lo splits); useful flops only"}}


# ---------------------------------------------------------------------------
# the CPU oracle (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def oracle_pair_sample(w: wl.Workload, seed: int = 0, extra: int = 0):
    """One (sequence, KV head) pair of the workload at full context, in the oracle
    (with room for `extra` more tokens)."""
    from oracle import kvq_oracle as ko
    rng = np.random.Generator(np.random.PCG64(seed))
    n = w.ctx
    k = rng.standard_normal((1, n, 1, w.head_dim), dtype=np.float32)
    v = rng.standard_normal((1, n, 1, w.head_dim), dtype=np.float32)
    k[..., rng.choice(w.head_dim, w.n_outliers, replace=False)] *= 20
    v[..., rng.choice(w.head_dim, w.n_outliers, replace=False)] *= 20
    k = wl.round_bf16(k) if w.dtype == "bf16" else k
    v = wl.round_bf16(v) if w.dtype == "bf16" else v
    rot = ko.rotation_enabled(w.head_dim)
    oc = ko.OracleCache(1, 1, w.head_dim, w.max_ctx(extra), w.tail_len, w.k_type, w.v_type, rot, rot)
    oc.append(k, v)
    q = rng.standard_normal((1, w.group, w.head_dim)).astype(np.float32)
    # one KV head's share: packed body + bf16 tail + q/out (bf16) of its query heads
    nbytes = (max(0, n - w.tail_len) * token_bytes(w) + min(n, w.tail_len) * 4 * w.head_dim
              + w.group * w.head_dim * 4)
    return oc, q, nbytes


def pair_step_bytes(w: wl.Workload, n: int, n_new: int) -> int:
    """One (sequence, KV head) pair's share of a step's algorithmic bytes: its decode
    at n tokens (packed body, bf16 tail, q / out of its query heads) and its append of
    n_new tokens.  For a batch whose sequences all hold n tokens, the pairs' shares add
    up to decode_bytes + append_bytes."""
    pairs = w.batch * w.n_kv_heads
    return (max(0, n - w.tail_len) * token_bytes(w) + min(n, w.tail_len) * 4 * w.head_dim
            + w.group * w.head_dim * 4 + append_bytes(w, n_new) // pairs)


def cpu_baseline(w: wl.Workload, budget_s: float = 15.0):
    from oracle import kvq_oracle as ko
    oc, q, nbytes = oracle_pair_sample(w)
    times = []
    t_all = time.perf_counter()
    while True:
        t0 = time.perf_counter()
        ko.decode_attention(oc, q)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_all > budget_s or len(times) >= 120:
            break
    per = statistics.median(times)
    # the write path too: the oracle appending one token per sequence to every KV head of the
    # workload (the decode step's append), rotation in float64 and float32 quantizers
    rng = np.random.Generator(np.random.PCG64(1))
    rot = ko.rotation_enabled(w.head_dim)
    oa = ko.OracleCache(w.batch, w.n_kv_heads, w.head_dim, 64, min(w.tail_len, 64), w.k_type, w.v_type, rot, rot)
    x = rng.standard_normal((w.batch, 1, w.n_kv_heads, w.head_dim)).astype(np.float32)
    at = []
    for _ in range(20):
        t0 = time.perf_counter()
        oa.append(x, x)
        at.append(time.perf_counter() - t0)
    app = statistics.median(at)
    return {"value": round(nbytes / per / 1e9, 4), "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"decode attention of 1 of {w.batch * w.n_kv_heads} (sequence, KV head) pairs at "
                      f"{w.ctx} tokens ({w.group} query heads), float64 numpy, {len(times)} repetitions, "
                      f"median {per:.3f} s",
            "append": {"tokens_per_s": round(w.batch / app, 1), "ms_per_call": round(app * 1e3, 3),
                       "sample": f"oracle append of 1 token to each of {w.batch} sequences x {w.n_kv_heads} KV heads, "
                                 f"20 repetitions, median"},
            "threads_note": "numpy elementwise work is single-threaded; its BLAS products may use all cores"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import kvq_oracle as ko
    w = wl.WORKLOADS[args.workload]
    n_new = max(1, w.append_per_step)
    W, K = args.warmup, args.steps
    oc, q, _ = oracle_pair_sample(w, extra=(W + K) * n_new)
    # the step's new tokens of the sampled pair, drawn ahead of the timed region
    rng = np.random.Generator(np.random.PCG64(11))
    new = []
    for _ in range(W + K):
        kv = rng.standard_normal((2, 1, n_new, 1, w.head_dim), dtype=np.float32)
        new.append(wl.round_bf16(kv) if w.dtype == "bf16" else kv)
    pairs = w.batch * w.n_kv_heads
    def step(i):
        oc.append(new[i][0], new[i][1])
        ko.decode_attention(oc, q)

    for i in range(W):
        step(i)
    n_first = int(oc.seq_len[0]) + n_new
    t0 = time.perf_counter()
    for i in range(K):
        step(W + i)
    dt = (time.perf_counter() - t0) / K
    nbytes = sum(pair_step_bytes(w, n_first + i * n_new, n_new) for i in range(K)) / K
    val = round(nbytes / dt / 1e9, 4)
    sample = (f"each step: the append of {n_new} new token(s) and decode attention of 1 of {pairs} "
              f"(sequence, KV head) pairs at {w.ctx}+ tokens (its share of the step's bytes), float64 / "
              f"float32 numpy oracle")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": w.name, "batch": w.batch, "ctx": w.ctx,
                                            "q_heads": w.n_q_heads, "kv_heads": w.n_kv_heads,
                                            "head_dim": w.head_dim, "k_type": w.k_type, "v_type": w.v_type,
                                            "tail_len": w.tail_len, "append_per_step": max(1, w.append_per_step),
                                            "l2": config_l2_note(w),
                                            "parallelism": "single GPU"},
            "cpu_baseline": {"value": val, "unit": "GB/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=wl.HEADLINE,
                    choices=sorted(k for k, v in wl.WORKLOADS.items() if not v.prefill))
    ap.add_argument("--ctx", type=int, default=0,
                    help="context length override (a smaller case of the same workload, e.g. for ncu captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prompt-workload measurement")
    ap.add_argument("--no-format-pairs", action="store_true",
                    help="skip the decode measurement with the q4_1 / q5_1 format pairs")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the decode measurement of the other workloads (d=64 ctx 256, GQA 16/8 ctx 4k, "
                         "ragged batch of 32)")
    ap.add_argument("--prefill-only", action="store_true",
                    help="run only the prompt-workload measurement (bulk append + prefill attention) and print "
                         "its record; for profiling the bulk write and prefill kernels")
    ap.add_argument("--configs-only", action="store_true",
                    help="run only the decode measurement of the other workloads (d=64 ctx 256, GQA 16/8 ctx "
                         "4k, ragged batch of 32) and print their records; for profiling those launches")
    ap.add_argument("--load-s", type=float, default=1.2,
                    help="seconds of extra decode load inside the clock-sampling window")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill_only:
        import torch
        from rotated_bit_kv_kvq_gb300 import kvq
        print(json.dumps({"prefill": run_prefill_bench(torch, kvq, args.steps, args.warmup)}), flush=True)
    elif args.configs_only:
        import torch
        from rotated_bit_kv_kvq_gb300 import kvq
        print(json.dumps({"configs": run_config_legs(torch, kvq, measured_peaks()[0])}), flush=True)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

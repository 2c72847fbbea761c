"""Benchmark of the batched paged-attention hot path on GB300.

One step = one pass of the whole path over one batch resident in HBM:
slot mapping -> scatter of the step's new K/V rows into the paged pool -> attention
(varlen: validation + plan, the tcgen05 prefill kernel for prefill chunks and the warp-MMA
kernel for decode tokens; split-KV: validation, partials, log-sum-exp reduction).  The
default workload is the 64-sequence decode batch with the Llama-3-8B attention shape
(H 32, Hkv 8, D 128, bf16, contexts U{512..4096}); its K/V (~600 MB per step) is larger
than L2, so no flush is needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 2|3|4|5] [--impl reference]

Prints one JSON line.  `value` is whole-job K/V GB/s (algorithmic K/V bytes the attention
reads per step, summed over ranks, divided by the slowest rank's time).  The line also
carries secondary per-class measurements of the other workloads (prefill-chunk TFLOP/s of
the mixed batch against the bf16 tensor peak, its decode GB/s, split-KV and shared-prefix
GB/s) unless --no-secondary.  With --gpus N > 1 (under torchrun) every rank runs an
independent replica ("replicas only": the path needs no exchange between GPUs).
--impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode KV GB/s (% HBM peak); mixed-batch prefill TFLOP/s; tokens/s"
KERNEL_SOURCES = {"k_mma16": "paged_kv_cache_31_gb300/csrc/k_decode_mma.cu",
                  "k_mma16_fp8": "paged_kv_cache_31_gb300/csrc/k_decode_mma.cu",
                  "k_tc_prefill": "paged_kv_cache_31_gb300/csrc/k_prefill_tc.cu",
                  "k_tc_prefill_fp8": "paged_kv_cache_31_gb300/csrc/k_prefill_tc.cu"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=2, choices=[2, 3, 4, 5])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--reference-seconds", type=float, default=120.0,
                    help="--impl reference: wall time all its steps together take, about")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="wall-time budget of the CPU oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--secondary-steps", type=int, default=30)
    ap.add_argument("--case", default="bench",
                    choices=["bench", "prefill-chunks", "prefill-chunks-fp8", "decode-fp8",
                             "splitkv", "shared-prefix", "tiny", "decode"],
                    help="a single timed case for profiling: prefill-chunks (the attention "
                         "call on the mixed batch's prefill chunks, own pool), decode-fp8 (the "
                         "decode batch over fp8 pools), splitkv (the long-context split-KV "
                         "call), shared-prefix (the fork batch's attention call), tiny (the "
                         "fp32 tiny mixed batch), decode (the decode batch's attention call), "
                         "prefill-chunks-fp8 (the prefill chunks over e4m3 pools)")
    ap.add_argument("--min-timed-ms", type=float, default=1000.0,
                    help="the timed loop of --steps steps is repeated until the repeats "
                         "together take at least this long (at least 5 repeats)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------
# ranks


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def aggregate(local_ms: float, units_per_rank: float, world: int, group=None):
    """Slowest rank's time and the whole-job throughput: units of all ranks / that time.
    Collective only when world > 1."""
    ms = local_ms
    if world > 1:
        import torch
        import torch.distributed as dist

        t = torch.tensor([local_ms], dtype=torch.float64)
        if dist.get_backend(group) == "nccl":
            t = t.cuda()
        dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
        ms = float(t.item())
    return ms, units_per_rank * world / (ms * 1e-3)


# ------------------------------------------------------------------------------------------
# workload accounting (algorithmic units, independent of the kernels)


def _ranges(w):
    qsl = w.query_start_loc.cpu().tolist()
    pos = w.positions.cpu().tolist()
    for s, n in enumerate(w.seq_lens_list):
        for t in range(qsl[s], qsl[s + 1]):
            e = pos[t] + 1 if w.causal else n
            b = max(0, e - w.sliding_window) if w.sliding_window > 0 else 0
            yield s, b, e


def kv_bytes(w, elem_bytes=None) -> int:
    """K and V bytes the attention must read: every visible (position, kv head) row once per
    sequence (the union of its tokens' visible ranges).  elem_bytes: the pool's element size
    when it differs from w.dtype's (1 for fp8 pools)."""
    esz = elem_bytes or (2 if str(w.dtype).endswith("bfloat16") else 4)
    row = w.num_kv_heads * w.head_dim * esz * 2
    span = {}
    for s, b, e in _ranges(w):
        lo, hi = span.get(s, (b, e))
        span[s] = (min(lo, b), max(hi, e))
    return sum((hi - lo) * row for lo, hi in span.values())


def attn_flops(w) -> int:
    """4 * D * H per visible (query token, key) pair: QK^T and PV multiply-adds."""
    return 4 * w.head_dim * w.num_heads * sum(e - b for _, b, e in _ranges(w))


def launches(w, varlen: bool) -> int:
    """Kernels of the library launched by one step: slot mapping + scatter (one kernel for up
    to 2048 tokens and 2047 sequences, else slot mapping, slot check and scatter), then
    validate+plan, the tcgen05 kernel when a sequence can exceed 64 query rows per kv head
    (the library's own rule) and the warp-MMA kernel; or, split-KV, validation, partials and
    reduction."""
    T, S, G = w.num_tokens, w.num_seqs, w.group
    cache = 1 if (T <= 2048 and S <= 2047) else 3
    if not varlen:
        return cache + 3
    tc = str(w.dtype).endswith("bfloat16") and w.head_dim == 128 and 128 % G == 0 and \
        (T - S + 1) * G > 64
    return cache + 2 + (1 if tc else 0)


# ------------------------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.out = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), float(parts[2]), float(parts[3]),
                             parts[4:8]))
            except ValueError:
                continue
        busy = [r for r in rows if r[3] > 0] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in busy for i, v in enumerate(r[4]) if v == "Active"})
        return {"sm_mhz": statistics.median(r[0] for r in busy) if busy else None,
                "sm_max_mhz": max(r[1] for r in busy) if busy else None,
                "power_w_max": max(r[2] for r in busy) if busy else None,
                "samples": len(busy), "reasons": reasons}


# ------------------------------------------------------------------------------------------
# measured peaks and ncu traffic


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "kind": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "kind": "fallback"}


def ncu_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch of `kernel` from the committed ncu summary, or None
    when there is none or the kernel source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{kernel}/{workload}")
    if not e:
        return None
    with open(os.path.join(ROOT, KERNEL_SOURCES[kernel]), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return e.get("bytes_per_launch") if e.get("source_sha") == sha else None


# ------------------------------------------------------------------------------------------
# the CPU oracle (reference arm and cpu_baseline)


def time_oracle(w, budget_s: float):
    """Run the oracle on the whole batch repeatedly for about budget_s seconds of wall time
    (at least once).  Returns (seconds per batch, batches run, threads)."""
    import oracle

    oracle.build()
    q, kb, vb = w.q.cpu(), w.k_blocks.cpu(), w.v_blocks.cpu()
    meta = [w.query_start_loc.cpu(), w.seq_lens.cpu(), w.positions.cpu(), w.block_tables.cpu()]
    n, t0 = 0, time.perf_counter()
    while True:
        st, _, _ = oracle.varlen_attention(q, kb, vb, *meta, w.scale, causal=w.causal,
                                           sliding_window=w.sliding_window)
        assert st == oracle.OK
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return el / n, n, oracle.num_threads()


def run_reference(args, w):
    """The reference arm: the CPU oracle on the host cores, --warmup untimed and --steps timed
    steps.  A step is one oracle pass over a bounded sample of the batch, its first n
    sequences, n sized from one calibration pass over the whole batch so that all the steps
    together take about --reference-seconds."""
    import oracle

    from paged_kv_cache_31_gb300 import workloads

    oracle.build()

    def one_pass(x):
        st, _, _ = oracle.varlen_attention(x.q.cpu(), x.k_blocks.cpu(), x.v_blocks.cpu(),
                                           x.query_start_loc.cpu(), x.seq_lens.cpu(),
                                           x.positions.cpu(), x.block_tables.cpu(), x.scale,
                                           causal=x.causal, sliding_window=x.sliding_window)
        assert st == oracle.OK

    t0 = time.perf_counter()
    one_pass(w)
    t_full = time.perf_counter() - t0
    per_step = args.reference_seconds / max(1, args.steps + args.warmup)
    n = w.num_seqs if t_full <= per_step else max(1, int(w.num_seqs * per_step / t_full))
    x = w if n == w.num_seqs else workloads.subset(w, list(range(n)), name=w.name)
    for _ in range(args.warmup):
        one_pass(x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_pass(x)
    per = (time.perf_counter() - t0) / max(1, args.steps)
    value = kv_bytes(x) / per / 1e9
    sample = (f"the whole {w.name} batch per step" if n == w.num_seqs else
              f"its first {n} of {w.num_seqs} sequences per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": {"workload": w.name, "num_seqs": w.num_seqs,
                                        "seed": args.seed},
        "tokens_per_s": x.num_tokens / per,
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# the GPU arm


class Runner:
    """Device buffers of one workload and the library calls of its step."""

    def __init__(self, pa, w, bitwise=False):
        import torch

        self.pa, self.w, self.bitwise = pa, w, bitwise
        self.varlen = not w.partition_size
        self.out = torch.empty_like(w.q)
        self.slots = torch.empty(w.num_tokens, dtype=torch.int32, device=w.q.device)
        self.ws = pa.workspace_for(w.q, w.k_blocks, w.query_start_loc, w.block_tables)
        if not self.varlen:
            S, H, D, P = w.num_seqs, w.num_heads, w.head_dim, w.max_partitions()
            self.ml = torch.empty((S, H, P), device=w.q.device)
            self.es = torch.empty((S, H, P), device=w.q.device)
            self.to = torch.empty((S, H, P, D), device=w.q.device)

    def cache(self, m=None):
        """Slot mapping and scatter of the new tokens' K/V (one launch for decode batches)."""
        w, pa = self.w, self.pa
        m = m or {}
        pa.pa_slot_mapping_and_cache(m.get("k_new", w.k_new), m.get("v_new", w.v_new),
                                     w.k_blocks, w.v_blocks,
                                     m.get("query_start_loc", w.query_start_loc),
                                     m.get("positions", w.positions),
                                     m.get("block_tables", w.block_tables), out=self.slots)

    def attention(self, m=None):
        w, pa = self.w, self.pa
        m = m or {}
        q = m.get("q", w.q)
        out = m.get("out", self.out)
        if self.varlen:
            pa.pa_varlen_forward(q, w.k_blocks, w.v_blocks, out,
                                 m.get("query_start_loc", w.query_start_loc),
                                 m.get("seq_lens", w.seq_lens), m.get("positions", w.positions),
                                 m.get("block_tables", w.block_tables), w.scale, causal=w.causal,
                                 sliding_window=w.sliding_window, workspace=self.ws,
                                 bitwise=self.bitwise)
        else:
            pa.pa_decode_splitkv(q, w.k_blocks, w.v_blocks, out, self.ml, self.es, self.to,
                                 m.get("seq_lens", w.seq_lens),
                                 m.get("block_tables", w.block_tables), w.scale,
                                 w.partition_size, w.sliding_window)

    def step(self, m=None):
        """One step: the new tokens' K/V into the cache, then attention (varlen: one library
        call, whose scatter overlaps the attention's planning kernel)."""
        if not self.varlen:
            self.cache(m)
            self.attention(m)
            return
        w, pa = self.w, self.pa
        m = m or {}
        pa.pa_cache_and_attend(m.get("k_new", w.k_new), m.get("v_new", w.v_new),
                               m.get("q", w.q), w.k_blocks, w.v_blocks, m.get("out", self.out),
                               m.get("query_start_loc", w.query_start_loc),
                               m.get("seq_lens", w.seq_lens), m.get("positions", w.positions),
                               m.get("block_tables", w.block_tables), w.scale, causal=w.causal,
                               sliding_window=w.sliding_window, workspace=self.ws,
                               slot_mapping=self.slots)


def time_calls(fn, n, stream, flush=None):
    """Mean ms per call of fn over n calls, timed with CUDA events on `stream`.  With `flush`
    (two buffers larger than L2) every call is timed on its own after overwriting the first
    buffer and then reading the second: no call finds the previous one's inputs in L2, and
    the flush's dirty lines are written back before the timed call, not inside it."""
    import torch

    if flush is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    wbuf, rbuf = flush
    for a, b in ev:
        wbuf.add_(1)
        rbuf.amax()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / n


def time_repeats(fn, steps, stream, min_total_ms, min_reps=5, max_reps=2000):
    """Repeat a timed loop of exactly `steps` calls (CUDA events on `stream`, synchronised
    after each loop) until the loops together took min_total_ms, at least min_reps times.
    Returns the per-call ms of every repeat."""
    out, total = [], 0.0
    while len(out) < max_reps and (len(out) < min_reps or total < min_total_ms):
        ms = time_calls(fn, steps, stream)
        out.append(ms)
        total += ms * steps
    return out


def spread(xs):
    """Median and range of repeat times (ms)."""
    ys = sorted(xs)
    return {"repeats": len(ys), "median_ms": statistics.median(ys), "min_ms": ys[0],
            "max_ms": ys[-1]}


def l2_flush_buffer(dev):
    """Two buffers of 256 MB, each about twice the GB300's L2: one to overwrite, one to read."""
    import torch

    return (torch.zeros(64 << 20, dtype=torch.float32, device=dev),
            torch.zeros(64 << 20, dtype=torch.float32, device=dev))


def prefill_back_to_back(pa, dev, args, peaks, stream, n, copies=6):
    """The prefill chunks as consecutive calls of a serving loop: `copies` copies of the
    workload's inputs (q, pools, output; together several times L2) taken in turn, with no
    flush between the calls.  No call finds its inputs in L2, and, as between the steps of a
    serving loop, each call's planner overlaps the previous call's tail."""
    import dataclasses

    import torch

    from paged_kv_cache_31_gb300 import workloads

    base = workloads.prefill_chunks(seed=args.seed, device=dev)
    runners = []
    for _ in range(copies):
        w = dataclasses.replace(base, q=base.q.clone(), k_blocks=base.k_blocks.clone(),
                                v_blocks=base.v_blocks.clone())
        runners.append(Runner(pa, w))
    per_copy = sum(t.numel() * t.element_size()
                   for t in (base.q, base.k_blocks, base.v_blocks, runners[0].out))
    for r in runners:
        r.attention()
        r.attention()
    nxt = [0]

    def call():
        runners[nxt[0]].attention()
        nxt[0] = (nxt[0] + 1) % copies

    ms = time_calls(call, n * copies, stream)
    fl = attn_flops(base)
    assert pa.pa_device_status() == pa.PA_OK
    return {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
            "frac_of_bf16_peak": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "l2": f"{copies} copies of the inputs ({copies * per_copy / 1e6:.0f} MB, "
                  "larger than L2) taken in turn, calls back to back"}


def fp8_decode(pa, dev, args, peaks, stream, n):
    """The decode batch over fp8 (e4m3) pools with dequantisation scales: half the K/V bytes
    of the bf16 batch, 303 MB of codes (larger than L2, so no flush)."""
    import torch

    from paged_kv_cache_31_gb300 import workloads

    w2 = workloads.named(2, seed=args.seed, device=dev)
    kb8, vb8 = workloads.fp8_pools(w2)
    out2 = torch.empty_like(w2.q)
    ws2 = pa.workspace_for(w2.q, kb8, w2.query_start_loc, w2.block_tables)
    # the same pools with one dequantisation scale per kv head, and one factor per (pool block,
    # kv head) (device arrays)
    hs = torch.full((w2.num_kv_heads,), 0.125, device=dev)
    bs = torch.full((kb8.shape[0], w2.num_kv_heads), 0.125, device=dev)

    def call(per_head=False, per_block=False):
        kw = (dict(k_scales=hs, v_scales=hs) if per_head
              else dict(k_block_scales=bs, v_block_scales=bs) if per_block
              else dict(k_scale=0.125, v_scale=0.125))
        pa.pa_varlen_forward(w2.q, kb8, vb8, out2, w2.query_start_loc, w2.seq_lens,
                             w2.positions, w2.block_tables, w2.scale, workspace=ws2, **kw)

    for _ in range(max(3, args.warmup)):
        call()
        call(True)
        call(False, True)
    ms = time_calls(call, n, stream)
    ms_h = time_calls(lambda: call(True), n, stream)
    ms_b = time_calls(lambda: call(False, True), n, stream)
    assert pa.pa_device_status() == pa.PA_OK
    kv = kv_bytes(w2, elem_bytes=1)
    name = w2.name + "-fp8"
    return {"workload": name, "kv_bytes": kv, "ms": ms, "gbs": kv / (ms * 1e-3) / 1e9,
            "frac_of_hbm": kv / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "l2": "inputs (pools of ~300 MB) larger than L2",
            "traffic": ncu_traffic("k_mma16_fp8", name),
            "per_head_scales": {"ms": ms_h, "gbs": kv / (ms_h * 1e-3) / 1e9,
                                "frac_of_hbm": kv / (ms_h * 1e-3) / 1e9 / peaks["hbm_gbs"]},
            "per_block_scales": {"ms": ms_b, "gbs": kv / (ms_b * 1e-3) / 1e9,
                                 "frac_of_hbm": kv / (ms_b * 1e-3) / 1e9 / peaks["hbm_gbs"]}}


def fp8_prefill(pa, dev, args, peaks, stream, n):
    """The mixed batch's prefill chunks over e4m3 pools with dequantisation scales (the
    tcgen05 kernel widens the codes to f16 in shared memory), L2 flushed between calls."""
    import torch

    from paged_kv_cache_31_gb300 import workloads

    wp = workloads.prefill_chunks(seed=args.seed, device=dev)
    kb8, vb8 = workloads.fp8_pools(wp)
    out = torch.empty_like(wp.q)
    ws = pa.workspace_for(wp.q, kb8, wp.query_start_loc, wp.block_tables)

    def call():
        pa.pa_varlen_forward(wp.q, kb8, vb8, out, wp.query_start_loc, wp.seq_lens,
                             wp.positions, wp.block_tables, wp.scale,
                             sliding_window=wp.sliding_window, workspace=ws, k_scale=0.125,
                             v_scale=0.125)

    for _ in range(max(3, args.warmup)):
        call()
    ms = time_calls(call, n, stream, flush=l2_flush_buffer(dev))
    assert pa.pa_device_status() == pa.PA_OK
    fl = attn_flops(wp)
    # back to back, as prefill_back_to_back: copies of the inputs taken in turn, no flush
    copies = 8
    sets = [(wp.q.clone(), kb8.clone(), vb8.clone(), torch.empty_like(wp.q),
             pa.workspace_for(wp.q, kb8, wp.query_start_loc, wp.block_tables))
            for _ in range(copies)]
    per_copy = sum(t.numel() * t.element_size() for t in sets[0][:4])
    nxt = [0]

    def call_rr():
        q, k8, v8, o, w_s = sets[nxt[0]]
        nxt[0] = (nxt[0] + 1) % copies
        pa.pa_varlen_forward(q, k8, v8, o, wp.query_start_loc, wp.seq_lens, wp.positions,
                             wp.block_tables, wp.scale, sliding_window=wp.sliding_window,
                             workspace=w_s, k_scale=0.125, v_scale=0.125)

    for _ in range(2 * copies):
        call_rr()
    ms_b = time_calls(call_rr, n * copies, stream)
    assert pa.pa_device_status() == pa.PA_OK
    return {"workload": wp.name + "-fp8", "flops": fl, "ms": ms, "l2": "flushed between calls",
            "tflops": fl / (ms * 1e-3) / 1e12,
            "frac_of_bf16_peak": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "mma": "f16 x f16 (codes and q widened to f16), fp32 accumulation",
            "traffic": ncu_traffic("k_tc_prefill_fp8", wp.name + "-fp8"),
            "back_to_back": {"ms": ms_b, "tflops": fl / (ms_b * 1e-3) / 1e12,
                             "frac_of_bf16_peak": fl / (ms_b * 1e-3) / 1e12 / peaks["bf16_tflops"],
                             "l2": f"{copies} copies of the inputs ({copies * per_copy / 1e6:.0f} "
                                   "MB, larger than L2) taken in turn, calls back to back"}}


def secondary(pa, dev, args, peaks, stream):
    """Per-class measurements of the mixed batch (prefill chunks alone: TFLOP/s of the
    tcgen05 path; decode tokens alone: K/V GB/s), the long-context split-KV batch and the
    shared-prefix fork batch."""
    import torch

    from paged_kv_cache_31_gb300 import workloads

    res = {}
    n = args.secondary_steps
    w3 = workloads.named(3, seed=args.seed, device=dev)
    r3 = Runner(pa, w3)
    for _ in range(3):
        r3.step()
    full_ms = time_calls(r3.step, n, stream)
    dec = [s for s, q in enumerate(w3.q_lens_list) if q == 1]
    pre = [s for s, q in enumerate(w3.q_lens_list) if q > 1]
    wp, wd = workloads.subset(w3, pre, "prefill-chunks"), workloads.subset(w3, dec, "decode")
    rp, rd = Runner(pa, wp), Runner(pa, wd)
    for _ in range(3):
        rp.attention()
        rd.attention()
    flush = l2_flush_buffer(dev)
    p_ms = time_calls(rp.attention, n, stream, flush=flush)  # its K/V would fit in L2
    # the same chunks with PA_FLAG_BITWISE (warp-MMA kernel: decode and prefill agree bitwise)
    rb = Runner(pa, wp, bitwise=True)
    for _ in range(3):
        rb.attention()
    b_ms = time_calls(rb.attention, n, stream, flush=flush)
    d_ms = time_calls(rd.attention, n, stream)
    del flush
    fl, kvd = attn_flops(wp), kv_bytes(wd)
    res["mixed"] = {
        "workload": w3.name, "tokens_per_s": w3.num_tokens / (full_ms * 1e-3),
        "ms_per_step": full_ms,
        "prefill": {"tokens": wp.num_tokens, "flops": fl, "ms": p_ms,
                    "tflops": fl / (p_ms * 1e-3) / 1e12,
                    "frac_of_bf16_peak": fl / (p_ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                    "l2": "flushed between calls",
                    "bound": "tensor", "peak_tflops": peaks["bf16_tflops"],
                    "traffic": ncu_traffic("k_tc_prefill", wp.name),
                    "bitwise_flag": {"ms": b_ms, "tflops": fl / (b_ms * 1e-3) / 1e12,
                                     "kernel": "warp-MMA (PA_FLAG_BITWISE)"}},
        "decode": {"tokens": wd.num_tokens, "kv_bytes": kvd, "ms": d_ms,
                   "gbs": kvd / (d_ms * 1e-3) / 1e9,
                   "frac_of_hbm": kvd / (d_ms * 1e-3) / 1e9 / peaks["hbm_gbs"]},
    }
    assert pa.pa_device_status() == pa.PA_OK
    del w3, r3, wp, wd, rp, rd, rb
    torch.cuda.empty_cache()
    res["mixed"]["prefill"]["back_to_back"] = prefill_back_to_back(pa, dev, args, peaks,
                                                                   stream, n)
    torch.cuda.empty_cache()

    res["fp8_decode"] = fp8_decode(pa, dev, args, peaks, stream, n)
    torch.cuda.empty_cache()
    res["fp8_prefill"] = fp8_prefill(pa, dev, args, peaks, stream, n)
    torch.cuda.empty_cache()

    w4 = workloads.named(4, seed=args.seed, device=dev)
    r4 = Runner(pa, w4)
    for _ in range(3):
        r4.attention()
    ms4 = time_calls(r4.attention, max(5, n // 3), stream)
    kv4 = kv_bytes(w4)
    res["splitkv"] = {"workload": w4.name, "kv_bytes": kv4, "ms": ms4,
                      "gbs": kv4 / (ms4 * 1e-3) / 1e9,
                      "frac_of_hbm": kv4 / (ms4 * 1e-3) / 1e9 / peaks["hbm_gbs"],
                      "traffic_partials": ncu_traffic("k_mma16", w4.name)}
    assert pa.pa_device_status() == pa.PA_OK
    del w4, r4
    torch.cuda.empty_cache()

    w5 = workloads.named(5, seed=args.seed, device=dev)
    r5 = Runner(pa, w5)
    for _ in range(3):
        r5.attention()
    ms5 = time_calls(r5.attention, n, stream)
    kv5 = kv_bytes(w5)
    # bytes the decode kernel actually read from DRAM (shared blocks once, the rest through
    # L2), from the committed ncu capture of this call
    uniq = ncu_traffic("k_mma16", w5.name)
    res["shared_prefix"] = {"workload": w5.name, "logical_kv_bytes": kv5, "ms": ms5,
                            "logical_gbs": kv5 / (ms5 * 1e-3) / 1e9,
                            "dram_bytes": uniq,
                            "dram_gbs": None if uniq is None else uniq / (ms5 * 1e-3) / 1e9,
                            "tokens_per_s": w5.num_tokens / (ms5 * 1e-3)}
    assert pa.pa_device_status() == pa.PA_OK
    del w5, r5
    torch.cuda.empty_cache()

    # the tiny fp32 mixed batch: a latency figure (general kernel; far too small to load the
    # GPU), per attention call and per whole step
    w1 = workloads.named(1, seed=args.seed, device=dev)
    r1 = Runner(pa, w1)
    for _ in range(3):
        r1.step()
    ms1a = time_calls(r1.attention, n, stream)
    ms1s = time_calls(r1.step, n, stream)
    assert pa.pa_device_status() == pa.PA_OK
    res["tiny_mixed"] = {"workload": w1.name, "tokens": w1.num_tokens, "us_per_call": ms1a * 1e3,
                         "us_per_step": ms1s * 1e3, "dtype": "f32"}
    del w1, r1

    # the two-state merge of chunked-context prefill: 16384 query tokens x 32 heads x 128,
    # bf16 states with fp32 lse (410 MB moved, larger than L2, so no flush)
    T, H, D = 16384, 32, 128
    g = torch.Generator(device=dev).manual_seed(args.seed + 11)
    po = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    so = torch.randn((T, H, D), generator=g, device=dev).to(torch.bfloat16)
    pl = torch.randn((H, T), generator=g, device=dev) * 4
    sl = torch.randn((H, T), generator=g, device=dev) * 4
    mo, ml = torch.empty_like(po), torch.empty_like(pl)

    def merge():
        pa.pa_merge_attn_states(mo, ml, po, pl, so, sl)

    for _ in range(3):
        merge()
    msm = time_calls(merge, n, stream)
    assert pa.pa_device_status() == pa.PA_OK
    mb = 3 * T * H * D * 2 + 3 * H * T * 4
    res["merge_attn_states"] = {"workload": f"merge-{T}x{H}x{D}-bf16", "bytes": mb, "ms": msm,
                                "gbs": mb / (msm * 1e-3) / 1e9,
                                "frac_of_hbm": mb / (msm * 1e-3) / 1e9 / peaks["hbm_gbs"],
                                "l2": "states larger than L2, no flush"}
    del po, so, pl, sl, mo, ml
    return res


def main():
    args = parse()
    rank, world, local = dist_env()
    import torch

    from paged_kv_cache_31_gb300 import workloads

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, workloads.named(args.config, seed=args.seed, device="cpu"))
        return

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    group = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
    from paged_kv_cache_31_gb300 import binding as pa

    peaks = measured_peaks()
    if args.case == "prefill-chunks-fp8":
        print(json.dumps(dict(case="prefill-chunks-fp8",
                              **fp8_prefill(pa, dev, args, peaks, torch.cuda.current_stream(),
                                            args.steps))), flush=True)
        return
    if args.case == "decode-fp8":
        print(json.dumps(dict(case="decode-fp8", **fp8_decode(pa, dev, args, peaks,
                                                               torch.cuda.current_stream(),
                                                               args.steps))), flush=True)
        return
    if args.case in ("splitkv", "shared-prefix", "tiny", "decode"):
        w = workloads.named({"splitkv": 4, "shared-prefix": 5, "tiny": 1, "decode": 2}[args.case],
                            seed=args.seed, device=dev)
        r = Runner(pa, w)
        for _ in range(max(3, args.warmup)):
            r.attention()
        ms = time_calls(r.attention, args.steps, torch.cuda.current_stream())
        assert pa.pa_device_status() == pa.PA_OK
        kv = kv_bytes(w)
        print(json.dumps({"case": w.name, "kv_bytes": kv, "ms": ms,
                          "gbs": kv / (ms * 1e-3) / 1e9}), flush=True)
        return
    if args.case == "prefill-chunks":
        wp = workloads.prefill_chunks(seed=args.seed, device=dev)
        rp = Runner(pa, wp)
        for _ in range(max(3, args.warmup)):
            rp.attention()
        ms = time_calls(rp.attention, args.steps, torch.cuda.current_stream(),
                        flush=l2_flush_buffer(dev))
        assert pa.pa_device_status() == pa.PA_OK
        fl = attn_flops(wp)
        print(json.dumps({"case": wp.name, "flops": fl, "ms": ms, "l2": "flushed between calls",
                          "tflops": fl / (ms * 1e-3) / 1e12,
                          "frac_of_bf16_peak": fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]}),
              flush=True)
        return
    w = workloads.named(args.config, seed=args.seed, device=dev)
    kvb = kv_bytes(w)
    flops = attn_flops(w)
    T = w.num_tokens
    run = Runner(pa, w)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for _ in range(max(3, args.warmup)):
        run.step()
    torch.cuda.synchronize()
    assert pa.pa_device_status() == pa.PA_OK

    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler(f"GPU-{uuid}" if uuid is not None else local)
    with sampler:
        time.sleep(0.3)
        # ---- whole step, inputs resident in HBM: the loop of --steps steps, repeated
        barrier()
        torch.cuda.synchronize()
        step_reps = time_repeats(run.step, args.steps, stream, args.min_timed_ms)
        step_ms = statistics.median(step_reps)
        barrier()
        # ---- the attention call alone (the dominant kernels)
        attn_reps = time_repeats(run.attention, args.steps, stream, args.min_timed_ms / 2)
        attn_ms = statistics.median(attn_reps)

        # ---- end to end through the public API with host buffers: every step copies its
        # inputs (packed in one pinned buffer) to the device and its output back, on a copy
        # stream, double-buffered, so step i+1's input copy and step i's output copy overlap
        # step i's kernels, as a serving loop would run them
        names = ["q", "k_new", "v_new", "query_start_loc", "seq_lens", "positions", "block_tables"]
        src = {k: getattr(w, k).contiguous() for k in names}
        layout, off = {}, 0
        for k, t in src.items():
            nb = t.numel() * t.element_size()
            layout[k] = (off, nb)
            off = (off + nb + 255) // 256 * 256
        hbuf = torch.empty(off, dtype=torch.uint8).pin_memory()
        for k, t in src.items():
            o, nb = layout[k]
            hbuf[o:o + nb].copy_(t.cpu().reshape(-1).view(torch.uint8))
        stage = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]
        views = [{k: stage[i][o:o + nb].view(src[k].dtype).view(src[k].shape)
                  for k, (o, nb) in layout.items()} for i in range(2)]
        douts = [torch.empty_like(w.q) for _ in range(2)]
        for i in range(2):
            views[i]["out"] = douts[i]
        houts = [torch.empty(w.q.shape, dtype=w.q.dtype).pin_memory() for _ in range(2)]
        h2d = sum(nb for _, nb in layout.values())
        d2h = houts[0].numel() * houts[0].element_size()
        e2e_steps = args.steps  # per repeat, as the device-timed loop
        e2e_repeats = 5          # the same on every rank (each repeat ends at a barrier)
        cstream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]

        def prefetch(b):  # this step's inputs into staging buffer b, once its last user ended
            cstream.wait_event(done[b])
            with torch.cuda.stream(cstream):
                stage[b].copy_(hbuf, non_blocking=True)
            copied[b].record(cstream)

        def e2e_step(i):
            b = i & 1
            stream.wait_event(copied[b])
            run.step(views[b])
            done[b].record(stream)
            prefetch(b ^ 1)  # the next step's inputs, during this step's kernels
            cstream.wait_event(done[b])
            with torch.cuda.stream(cstream):
                houts[b].copy_(douts[b], non_blocking=True)  # this step's output to the host

        for b in range(2):
            done[b].record(stream)
        prefetch(0)
        for i in range(3):
            e2e_step(i)
        e2e_reps = []
        for _ in range(e2e_repeats):
            torch.cuda.synchronize()
            barrier()
            t0 = time.perf_counter()
            prefetch(0)
            for i in range(e2e_steps):
                e2e_step(i)
            torch.cuda.synchronize()
            e2e_reps.append((time.perf_counter() - t0) * 1e3 / e2e_steps)
            barrier()
        e2e_ms = statistics.median(e2e_reps)
        assert torch.equal(houts[(e2e_steps - 1) & 1].to(dev), run.out), "e2e output differs"
    assert pa.pa_device_status() == pa.PA_OK, "device status set during the timed region"
    clocks = sampler.summary()

    step_ms, value = aggregate(step_ms, kvb / 1e9, world, group)
    e2e_ms, e2e_value = aggregate(e2e_ms, kvb / 1e9, world, group)
    if rank != 0:
        return
    achieved = kvb / (attn_ms * 1e-3) / 1e9
    # the decode batch's attention kernel, and the split-KV partials kernel (the same
    # warp-MMA kernel in its split mode); ncu traffic is recorded per (kernel, workload)
    kernel = "k_mma16"
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "num_seqs": w.num_seqs, "num_tokens": T,
                   "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads,
                   "head_dim": w.head_dim, "block_size": w.block_size,
                   "sliding_window": w.sliding_window, "kv_bytes_per_step": kvb,
                   "attn_flops_per_step": flops, "seed": args.seed,
                   "l2": f"inputs larger than L2 ({kvb / 1e6:.0f} MB of K/V read per step)",
                   "parallelism": "replicas" if world > 1 else "single"},
        "tokens_per_s": T * world / (step_ms * 1e-3),
        "timing": {"step": spread(step_reps), "attention_call": spread(attn_reps),
                   "e2e_step": spread(e2e_reps), "steps_per_repeat": args.steps},
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches(w, run.varlen) * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": ncu_traffic(kernel, w.name),
                     "kernel": kernel,
                     "timed_as": "one library call: the validate+plan kernel (a few us, "
                                 "overlapped by programmatic dependent launch) and " + kernel,
                     "peak_kind": f"{peaks['kind']} hbm_gbs (copy)", "ms_per_launch": attn_ms},
    }
    if not args.no_secondary:
        line["secondary"] = secondary(pa, dev, args, peaks, stream)
    if not args.no_cpu_baseline:
        per, n, cores = time_oracle(w, args.cpu_seconds)
        line["cpu_baseline"] = {"value": kvb / per / 1e9, "unit": "GB/s", "cores": cores,
                                "kind": "oracle",
                                "sample": f"{n} passes of the whole {w.name} batch "
                                          f"({per:.2f} s each)"}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

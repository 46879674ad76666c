"""Benchmark of the sparse paged decode hot path.

One step = the three stages over one batch of the stress sparse decode
workload (64 request rows of 1, 4, 8 or 16 query tokens -- 496 rows, 13 of
them padding --, 64 q / 8 kv heads, head dim 128, one index head of dim 128,
seq_lens log-uniform in [256, 16384] over an 8192-page pool, top-64 blocks,
FP8-E4M3 K/V, heavy-tailed queries): msa_block_score -> msa_select_topk ->
paged_sparse_decode_attention, all through the C ABI.  --config 2 runs the
EAGLE-style verification decode (4 rows x 4 tokens, top-16), --config 3 the
dense paged decode (16 rows of 16384 tokens, every block) instead.

Printed (rank 0, one JSON line): query rows per second (a query row is one
non-padding query token with all its heads), the attention kernel's achieved
HBM bandwidth against the measured peak, the end-to-end rate through the same
calls with host buffers, and the CPU oracle's rate on a bounded sample (the
single-threaded oracle called from one host thread per core on disjoint query
rows, and from one thread).  The run fails (exit 3) if an attention call
recorded a device-side wait that timed out.

Timing: CUDA events on the launching stream around each step; between timed
steps a 256 MiB buffer is rewritten to flush the 129 MB L2, then a second
256 MiB buffer is read so that the flush's dirty lines are written back
before the step rather than during it (both outside the events); W warm-up
steps first.  Under torchrun each rank runs its own batch
(different seed) with no data exchange: weak scaling, max time over ranks.

With --config prefill the step is one fused prefill score-to-selection call
(msa_prefill_block_score) over the batched prefill sequences (8 x 512-token
chunks, query blocks of 64 tokens, 1 initial + 2 local blocks, top-32); its
roofline is the score FLOPs against the dense bf16 tensor peak.

With --config dense the step is instead one dense GQA attention call
(attention_sdpa) on a causal prefill chunk: 512 query tokens after 7680 cached
tokens, 64 q / 8 kv heads, head dim 128, bf16; its roofline is the call's
algorithmic FLOPs against the dense bf16 tensor peak.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C|dense|prefill] [--impl reference]
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from sparse_paged_decode_gb300 import workloads as W  # noqa: E402

METRIC = "decode query-rows/sec and achieved HBM GB/s vs ~8 TB/s (sparse paged decode)"
UNIT = "query-rows/s"
DENSE_METRIC = "dense GQA attention query-rows/sec (prefill chunk)"
PREFILL_METRIC = "fused prefill score-to-selection query-rows/sec (batched paged prefill)"
BS = 128
FLUSH_BYTES = 256 << 20


# -------------------------------------------------------------------- helpers

class TimedOutWait(RuntimeError):
    """An attention call's workspace status says a device-side wait gave up."""


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback 6.8 TB/s"


def measured_bf16_peak():
    """Dense bf16 tensor peak in TFLOP/s (burst: the score kernel is timed alone)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    return 1900.0, "fallback 1.9 PFLOP/s"


def score_flops(w):
    """Algorithmic FLOPs of one score call: every query token against every
    key it may see (below its seq_len), Di multiply-adds each, per index head."""
    lim = np.minimum(np.maximum(w.seq_lens.numpy().astype(np.int64), 0), w.NB * BS)
    return float(2 * int(lim.sum()) * w.Di * w.Hi)


def workload_desc(w):
    return {
        "workload": next((W.CONFIG_NAMES[k] for k, n in W.WORKLOAD_NAMES.items() if n == w.name), w.name),
        "requests": w.R, "query_rows": w.T, "valid_query_rows": w.n_valid_tokens,
        "tokens_per_request": w.tokens_per_request, "request_lengths": w.request_lengths,
        "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.D, "index_heads": w.Hi, "index_dim": w.Di,
        "block_size": w.block_size, "page_table_blocks": w.NB, "pool_pages": w.P, "top_k": w.K,
        "kv_dtype": (None if w.k_cache is None else "e4m3 (static scalar scales)"
                     if w.k_cache.dtype == torch.float8_e4m3fn else "bfloat16 (dense)"),
        "q_dtype": str(w.q.dtype).replace("torch.", "") if w.q is not None else None,
        "index_dtype": str(w.q_idx.dtype).replace("torch.", "") if w.q_idx is not None else None,
        "index_cache_dtype": (str(w.k_idx_cache.dtype).replace("torch.", "")
                              if w.k_idx_cache is not None else None),
        "l2": "flushed between timed steps (256 MiB rewrite, then a 256 MiB read that cleans the dirty lines; "
              "outside the events)",
    }


def fp8_attention_kernel(w):
    """Name of the tensor-core kernel the library's default picks for an FP8
    cache and bf16 queries: the query-rows kernel when the batch averages at
    least 48 query rows (tokens x q heads of one kv head) per request."""
    G = w.Hq // w.Hkv
    R = w.block_table.shape[0]
    return "attention_e4m3_rows_kernel" if w.T * G >= 48 * R else "attention_tc_kernel"


def attention_bytes(w, topk_np):
    """Algorithmic bytes of one attention launch: every selected (request, kv
    head, block) page of K and V read once for its valid tokens (query rows of
    one request share a page read), plus q, out, topk_idx and the page table."""
    kv = 0
    start = 0
    for r, n in enumerate(w.tokens_per_request):
        rows = range(start, start + n)
        start += n
        L = max((int(w.seq_lens[t]) for t in rows), default=0)
        for h in range(w.Hkv):
            blocks = set()
            for t in rows:
                if int(w.seq_lens[t]) <= 0:
                    continue
                lim = min(int(w.seq_lens[t]), w.NB * BS)
                ids = range(w.NB) if topk_np is None else topk_np[min(h, topk_np.shape[0] - 1), t]
                for b in ids:
                    b = int(b)
                    if 0 <= b < w.NB and b * BS < lim:
                        blocks.add(b)
            for b in blocks:
                valid = min(BS, min(L, w.NB * BS) - b * BS)
                kv += 2 * valid * w.D * w.k_cache.element_size()
    q_bytes = w.q.numel() * w.q.element_size()
    out_bytes = w.T * w.Hq * w.D * 2
    tk_bytes = 0 if topk_np is None else w.T * w.K * 4
    return kv + q_bytes + out_bytes + tk_bytes + w.block_table.numel() * 4 + 2 * w.T * 4


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while a region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY, "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- the CPU baseline

def host_cores():
    """Cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):  # pragma: no cover
        return os.cpu_count() or 1


def oracle_rate(w, budget_s=12.0, max_rows=None, threads=1):
    """The oracle's three stages, row by row, on a bounded sample of the
    workload's query rows; returns (rows/s, rows timed, seconds).

    With threads > 1 the single-threaded oracle is called from that many host
    threads at once, each taking the next untimed row (ctypes releases the
    interpreter lock inside the call and the oracle keeps no state between
    calls); every thread stops taking rows once the budget is spent, and the
    rate is the rows finished over the wall time until the last one ends."""
    import oracle

    o = oracle.default()
    rows = [t for t in range(w.T) if int(w.seq_lens[t]) > 0]
    lock = threading.Lock()
    state = {"next": 0, "done": 0}
    t0 = time.perf_counter()

    def one(t):
        idx = torch.tensor([t])
        s = o.block_score(w.q_idx[idx], w.k_idx_cache, w.block_table, w.req_idx[idx], w.seq_lens[idx],
                          float(np.float32(w.idx_scale)))
        tk = o.select_topk(s, w.K)
        if w.q is not None:  # prefill score-to-selection has no attention stage
            o.paged_attention(w.q[idx], w.k_cache, w.v_cache, w.block_table, w.req_idx[idx], w.seq_lens[idx], tk,
                              float(np.float32(w.sm_scale)), float(np.float32(w.k_scale)),
                              float(np.float32(w.v_scale)))

    def worker():
        while True:
            with lock:
                if (state["next"] >= len(rows) or time.perf_counter() - t0 >= budget_s
                        or (max_rows and state["next"] >= max_rows)):
                    return
                t = rows[state["next"]]
                state["next"] += 1
            one(t)
            with lock:
                state["done"] += 1

    if threads <= 1:
        worker()
    else:
        pool = [threading.Thread(target=worker) for _ in range(threads)]
        for th in pool:
            th.start()
        for th in pool:
            th.join()
    dt = time.perf_counter() - t0
    return state["done"] / dt, state["done"], dt


def cpu_baseline_record(rate_fn, what, budget_s):
    """The oracle's rate on the host: all cores (one thread per core, the
    reported value) and one core (context)."""
    cores = host_cores()
    rate, n, dt = rate_fn(budget_s, cores)
    rate1, n1, dt1 = rate_fn(budget_s / 2, 1)
    return {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "%d %s through the single-threaded oracle (plain C, fp64) called from %d host threads "
                      "on disjoint rows, %.1f s" % (n, what, cores, dt),
            "one_core": {"value": rate1, "cores": 1, "sample": "%d %s on one thread, %.1f s" % (n1, what, dt1)}}


# ------------------------------------------------------------ replicas
# The path has no exchange step: N ranks run N independent batches (weak
# scaling).  These are the only places the ranks meet.

def batch_seed(config, rank):
    """Seed of a rank's synthetic batch: every rank gets its own inputs."""
    return 1000 + config + 97 * rank


def max_over_ranks(values, world, device):
    """Element-wise maximum of per-rank timings (the slowest rank sets the
    job's time)."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t]


def job_rate(rows_per_rank, world, steps, total_ms):
    """Whole-job throughput: the query rows all ranks processed over the
    slowest rank's time."""
    return rows_per_rank * world * steps / (total_ms / 1e3)


def make_workload(args, seed):
    """The configuration's batch; with --index-cache e4m3 its index cache is
    stored as FP8-E4M3 (scale folded into idx_scale)."""
    w = W.config(args.config, seed=seed, kv_dtype=args.kv_cache)
    return W.with_fp8_index(w) if args.index_cache == "e4m3" and w.k_idx_cache is not None else w


# --------------------------------------------------------------------- arms

def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = make_workload(args, 1000 + args.config)
    cores = host_cores()
    per_step_budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rate(w, budget_s=per_step_budget / 4, max_rows=1)
    rates, rows, secs = [], 0, 0.0
    for _ in range(args.steps):
        r, n, dt = oracle_rate(w, budget_s=per_step_budget, threads=cores)
        rates.append(r)
        rows += n
        secs += dt
    value = rows / secs
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_desc(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d query rows of the workload through the oracle's three stages "
                                   "(single-threaded C, fp64, called from %d host threads on disjoint rows), "
                                   "%.1f s per step" % (rows, cores, per_step_budget)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


ATTENTION_POLICY = {"auto": 0, "general": 1, "lanes": 2, "rows": 3}


def run_gpu(args, rank, world, local_rank):
    import sparse_paged_decode_gb300 as spd

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    spd.set_kernel_policy(3, ATTENTION_POLICY[args.attention_kernel])
    w = make_workload(args, batch_seed(args.config, rank))
    g = w.to(dev)
    # the step's per-call inputs live in one device buffer (each tensor a
    # 256-byte aligned view), so the end-to-end run stages them with a
    # single host-to-device copy
    in_names = [k for k in ("q", "q_idx", "block_table", "seq_lens", "req_idx") if getattr(w, k) is not None]
    offs, total_in = {}, 0
    for k in in_names:
        t = getattr(w, k)
        offs[k] = total_in
        total_in += (t.numel() * t.element_size() + 255) // 256 * 256
    dev_pack = torch.zeros(total_in, dtype=torch.uint8, device=dev)
    host_pack = torch.zeros(total_in, dtype=torch.uint8).pin_memory()
    for k in in_names:
        t = getattr(w, k).contiguous()
        nb = t.numel() * t.element_size()
        host_pack[offs[k]:offs[k] + nb].copy_(t.view(-1).view(torch.uint8))
        view = dev_pack[offs[k]:offs[k] + nb].view(t.dtype).view(t.shape)
        view.copy_(getattr(g, k))
        setattr(g, k, view)
    T, NB, K = w.T, w.NB, max(w.K, 1)
    scores = torch.empty((w.Hi, T, NB), device=dev)
    topk = torch.empty((w.Hi, T, K), dtype=torch.int32, device=dev)
    prefill = w.q is None  # prefill score-to-selection: no attention stage
    out = ws = None
    if not prefill:
        out = torch.empty((T, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(spd.decode_workspace_bytes(T, w.Hq, w.Hkv, w.D, NB), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    clean_sum = torch.empty((), dtype=torch.int64, device=dev)

    def flush_l2(i):
        # rewrite 256 MiB (evicts every input), then read another 256 MiB so
        # the rewrite's dirty lines are written back here, not in the step
        flush.fill_(i & 0xFF)
        torch.sum(clean, 0, dtype=torch.int64, out=clean_sum)

    stream = torch.cuda.current_stream(dev)
    dense = w.dense

    def attention(gg):
        if dense:
            spd.paged_decode_attention(gg.q, gg.k_cache, gg.v_cache, gg.block_table, gg.seq_lens, gg.req_idx, out,
                                       gg.sm_scale, BS, gg.k_scale, gg.v_scale, ws)
        else:
            spd.paged_sparse_decode_attention(gg.q, gg.k_cache, gg.v_cache, gg.block_table, gg.seq_lens,
                                              gg.req_idx, topk.expand(w.Hkv, -1, -1), out, gg.sm_scale, BS,
                                              gg.k_scale, gg.v_scale, ws)

    def score_call(gg):
        spd.msa_block_score(gg.q_idx, gg.k_idx_cache, gg.block_table, gg.seq_lens, gg.req_idx, BS, scores,
                            gg.idx_scale)

    # the call the roofline is taken on: the attention call for decode, the
    # score call for prefill
    timed = score_call if prefill else attention

    def step(gg, evs=None):
        if prefill:
            if evs is not None:
                evs[0].record(stream)
            score_call(gg)
            if evs is not None:
                evs[1].record(stream)
            spd.msa_select_topk(scores, topk)
            return
        if not dense:
            score_call(gg)
            spd.msa_select_topk(scores, topk)
        if evs is not None:
            evs[0].record(stream)
        attention(gg)
        if evs is not None:
            evs[1].record(stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step(g)
    torch.cuda.synchronize(dev)

    # the step runs as one captured CUDA graph, as a serving engine runs it:
    # kernel-to-kernel gaps are the GPU's own, not Python's launch latency
    graph = graph_attn = None
    if not args.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(g)
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            step(g)
        torch.cuda.synchronize(dev)
        # the attention call alone (its three kernels; the score call for
        # prefill), for the roofline
        graph_attn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_attn, stream=side):
            timed(g)
        torch.cuda.synchronize(dev)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.25)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    attn = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    n0 = spd.launch_count()
    step(g)
    torch.cuda.synchronize(dev)
    launches_per_step = spd.launch_count() - n0
    launches0 = spd.launch_count()
    for i in range(args.steps):
        flush_l2(i)
        starts[i].record(stream)
        if graph is not None:
            graph.replay()
        else:
            step(g, attn[i])
        ends[i].record(stream)
    torch.cuda.synchronize(dev)
    launches = spd.launch_count() - launches0
    if graph is not None:
        # a replay enqueues the captured kernels without calling the library
        launches = launches_per_step * args.steps
        # the attention call's device time: its own graph replayed between
        # events on the same stream, L2 flushed before each
        for i in range(args.steps):
            flush_l2(i)
            attn[i][0].record(stream)
            graph_attn.replay()
            attn[i][1].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    attn_ms = [a.elapsed_time(b) for a, b in attn]
    total_ms = sum(step_ms)

    # end to end through the same calls with host buffers: the step's inputs
    # (queries, index queries, page table, seq_lens, req_idx), packed in one
    # pinned buffer, copied in with one transfer, the attention output (the
    # top-k ids for prefill) copied back; caches stay resident
    result = topk if prefill else out
    host_out = torch.empty(result.shape, dtype=result.dtype).pin_memory()
    h2d = total_in
    d2h = host_out.numel() * host_out.element_size()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush_l2(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dev_pack.copy_(host_pack, non_blocking=True)
        if graph is not None:
            graph.replay()
        else:
            step(g)
        host_out.copy_(result, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    clocks = sampler.stop() if sampler else None
    # every attention call above left its status in the workspace: bit 0 =
    # a device-side wait timed out, so the timed outputs are not valid
    ws_status = spd.workspace_status(ws) if ws is not None else 0

    # max over ranks
    total_ms, e2e_total, bad = max_over_ranks([total_ms, sum(e2e_ms), float(ws_status != 0)], world, dev)
    if bad:
        raise TimedOutWait("an attention call recorded a device-side wait that timed out (workspace status %d)"
                           % ws_status)
    if rank != 0:
        return None

    value = job_rate(w.n_valid_tokens, world, args.steps, total_ms)
    e2e_value = job_rate(w.n_valid_tokens, world, args.steps, e2e_total)
    topk_np = None if dense else topk.cpu().numpy()
    attn_mean_s = statistics.mean(attn_ms) / 1e3
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "attention_traffic.json")
    if os.path.exists(tpath):
        with open(tpath) as f:
            tj = json.load(f)
        # a capture counts only while the attention call's sources are the
        # ones it was taken on
        for ent in tj.get("entries", []):
            if (ent.get("config") == args.config and ent.get("index_cache", "native") == args.index_cache
                    and ent.get("kv_cache", "e4m3") == args.kv_cache
                    and ent.get("attention_kernel", "auto") == args.attention_kernel
                    and ent.get("kernel_stamp") == _kernel_stamp(args.kv_cache)):
                traffic = ent.get("traffic_bytes_per_launch")
    if prefill:
        # the score call is a contraction: tensor-bound against the peak of
        # its operand type (bf16; an FP8 index cache takes the f8 product,
        # whose dense peak is nominally twice bf16's: 4.5 against 2.25 PF)
        flops = score_flops(w)
        achieved = flops / attn_mean_s / 1e12
        peak, peak_src = measured_bf16_peak()
        if w.k_idx_cache is not None and w.k_idx_cache.dtype == torch.float8_e4m3fn:
            peak, peak_src = 2.0 * peak, peak_src + " x 2 (nominal fp8 / bf16 dense ratio)"
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": None,
                    "kernel": "score call (score_tc_kernel; %s)" % ("graph replay" if graph is not None
                                                                      else "direct launches"),
                    "algorithmic_flops_per_launch": flops, "mean_launch_us": attn_mean_s * 1e6,
                    "peak_source": peak_src}
    else:
        abytes = attention_bytes(w, topk_np)
        achieved = abytes / attn_mean_s / 1e9
        peak, peak_src = measured_peaks()
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                    "traffic": traffic,
                    "kernel": "paged attention call (%s; %s)"
                              % ("general-layout kernel" if args.attention_kernel == "general" else
                                 "list planner, unit planner, " + (
                                     "attention_bf16_tc_kernel" if args.kv_cache == "bf16" else
                                     "attention_tc_kernel" if args.attention_kernel == "lanes" else
                                     "attention_e4m3_rows_kernel" if args.attention_kernel == "rows" else
                                     fp8_attention_kernel(w)),
                                 "graph replay" if graph is not None else "direct launches"),
                    "algorithmic_bytes_per_launch": abytes,
                    "mean_launch_us": attn_mean_s * 1e6, "peak_source": peak_src}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        wc = make_workload(args, 1000 + args.config)
        cpu = cpu_baseline_record(lambda b, n: oracle_rate(wc, budget_s=b, threads=n),
                                  "query rows of this workload (the oracle's %s)"
                                  % ("score and select stages" if prefill else "three stages"), args.cpu_seconds)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": (("e4m3 mma (index queries as two e4m3 terms)" if args.index_cache == "e4m3" else "bf16 mma")
                  + ", f32 accumulate") if prefill else ("e4m3/f16 mma, f32 accumulate"
                                                          if w.k_cache.dtype == torch.float8_e4m3fn
                                                          else "bf16 mma, f32 accumulate"),
        "data": "synthetic",
        "config": workload_desc(w),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "timed_as": "captured CUDA graph replay per step" if graph is not None else "direct launches per step",
        "clocks": clocks,
        "attention_ms_median": statistics.median(attn_ms),
        "step_ms_median": statistics.median(step_ms),
    }


# ------------------------------------------------- dense attention workload

def dense_flops(w):
    """Algorithmic FLOPs of one dense attention call: 2 D for the logit and
    2 D for the weighted value, per (query row, readable key) pair."""
    n_keys = 0
    for t in range(w.T):
        n = t + w.S - w.T + 1 if w.causal else w.S
        n_keys += max(0, min(w.S, n))
    return 4 * w.D * w.Hq * n_keys


def dense_oracle_rate(w, budget_s=12.0, max_tokens=None, threads=1):
    """The oracle on query tokens of the dense workload, one at a time (token
    t under the causal flag is non-causal attention over its first
    t + S - T + 1 keys), the longest rows first (a conservative rate), from
    `threads` host threads as in oracle_rate; returns (query tokens/s, tokens
    timed, seconds)."""
    import oracle

    o = oracle.default()
    order = list(range(w.T - 1, -1, -1))
    lock = threading.Lock()
    state = {"next": 0, "done": 0}
    t0 = time.perf_counter()

    def worker():
        while True:
            with lock:
                if (state["next"] >= len(order) or time.perf_counter() - t0 >= budget_s
                        or (max_tokens and state["next"] >= max_tokens)):
                    return
                t = order[state["next"]]
                state["next"] += 1
            n = t + w.S - w.T + 1 if w.causal else w.S
            o.sdpa(w.q[t:t + 1], w.k[:max(0, n)], w.v[:max(0, n)], float(np.float32(w.sm_scale)), False)
            with lock:
                state["done"] += 1

    pool = [threading.Thread(target=worker) for _ in range(max(1, threads))]
    for th in pool:
        th.start()
    for th in pool:
        th.join()
    dt = time.perf_counter() - t0
    return state["done"] / dt, state["done"], dt


def dense_desc(w):
    return {"workload": W.DENSE_NAME, "query_tokens": w.T, "keys": w.S, "Hq": w.Hq, "Hkv": w.Hkv,
            "head_dim": w.D, "causal": w.causal, "q_dtype": str(w.q.dtype)[6:], "kv_dtype": str(w.k.dtype)[6:],
            "out_dtype": "bfloat16",
            "l2": "flushed between timed steps (256 MiB rewrite, then a 256 MiB read that cleans the dirty "
                  "lines; outside the events)"}


def run_dense_reference(args, rank, world):
    if rank != 0:
        return None
    w = W.dense_prefill()
    cores = host_cores()
    per_step_budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        dense_oracle_rate(w, budget_s=per_step_budget / 4, max_tokens=1)
    rows, secs = 0, 0.0
    for _ in range(args.steps):
        _, n, dt = dense_oracle_rate(w, budget_s=per_step_budget, threads=cores)
        rows += n
        secs += dt
    value = rows / secs
    return {
        "impl": "reference", "metric": DENSE_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dense_desc(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d query tokens (all heads) of the chunk through the oracle (single-threaded "
                                   "C, fp64, called from %d host threads), %.1f s per step"
                                   % (rows, cores, per_step_budget)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_dense_gpu(args, rank, world, local_rank):
    import sparse_paged_decode_gb300 as spd

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = W.dense_prefill(seed=1006 + 97 * rank)
    g = w.to(dev)
    out = torch.empty((w.T, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    clean_sum = torch.empty((), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        torch.sum(clean, 0, dtype=torch.int64, out=clean_sum)

    def step():
        spd.attention_sdpa(g.q, g.k, g.v, out, w.sm_scale, w.causal)

    for i in range(args.warmup):
        flush_l2(i)
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.25)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    n0 = spd.launch_count()
    for i in range(args.steps):
        flush_l2(i)
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = spd.launch_count() - n0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]

    # end to end: the chunk's queries and its own 512 keys and values (the
    # prefix's stay resident, as in a KV cache) copied in from pinned host
    # memory, the output copied back
    new = slice(w.S - w.T, w.S)
    host_q = w.q.contiguous().pin_memory()
    host_k = w.k[new].contiguous().pin_memory()
    host_v = w.v[new].contiguous().pin_memory()
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (host_q, host_k, host_v))
    d2h = host_out.numel() * host_out.element_size()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush_l2(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.q.copy_(host_q, non_blocking=True)
        g.k[new].copy_(host_k, non_blocking=True)
        g.v[new].copy_(host_v, non_blocking=True)
        step()
        host_out.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    clocks = sampler.stop() if sampler else None

    total_ms, e2e_total = max_over_ranks([sum(step_ms), sum(e2e_ms)], world, dev)
    if rank != 0:
        return None
    value = job_rate(w.T, world, args.steps, total_ms)
    e2e_value = job_rate(w.T, world, args.steps, e2e_total)
    flops = dense_flops(w)
    mean_s = statistics.mean(step_ms) / 1e3
    achieved = flops / mean_s / 1e12
    peak, peak_src = measured_bf16_peak()
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline_record(lambda b, n: dense_oracle_rate(w, budget_s=b, threads=n),
                                  "query tokens (all heads; the longest rows) of the chunk", args.cpu_seconds)
    return {
        "metric": DENSE_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 mma (P bf16), f32 accumulate and softmax",
        "data": "synthetic", "config": dense_desc(w),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "sdpa_tc_kernel (direct launch)",
                     "algorithmic_flops_per_launch": flops, "mean_launch_us": mean_s * 1e6,
                     "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "timed_as": "direct launches per step",
        "clocks": clocks,
        "step_ms_median": statistics.median(step_ms),
    }


# ------------------------------------ fused prefill score-to-selection workload

def prefill_limits(pb):
    """(tokens, visible keys) of every query block of the batch."""
    cu, cub, pre, sl = (pb.cu_seqlens.tolist(), pb.cu_seqblocks_q.tolist(), pb.prefix_lens.tolist(),
                        pb.seq_lens.tolist())
    out = []
    for b in range(pb.B):
        for qb in range(cub[b + 1] - cub[b]):
            n_tok = max(0, min(pb.block_size_q, cu[b + 1] - cu[b] - qb * pb.block_size_q))
            L = max(0, min(pre[b] + qb * pb.block_size_q + 1, sl[b], pb.NB * BS))
            out.append((n_tok, L))
    return out


def prefill_flops(pb):
    """Algorithmic FLOPs of one fused prefill call: each query token of a
    query block against each key the block sees, Di multiply-adds, per index
    head."""
    return float(2 * pb.Di * pb.Hi * sum(n * L for n, L in prefill_limits(pb)))


def prefill_oracle_rate(pb, budget_s=12.0, max_rows=None, threads=1):
    """The oracle on the batch's query blocks, one at a time (each as a batch
    of its own: its tokens, with the block's first position as the prefix),
    from `threads` host threads as in oracle_rate, until the budget is spent;
    returns (query tokens/s, tokens timed, s)."""
    import oracle

    o = oracle.default()
    cu, cub, pre = pb.cu_seqlens.tolist(), pb.cu_seqblocks_q.tolist(), pb.prefix_lens.tolist()
    work = [(b, qb) for b in range(pb.B) for qb in range(cub[b + 1] - cub[b])]
    lock = threading.Lock()
    state = {"next": 0, "done": 0}
    t0 = time.perf_counter()

    def worker():
        while True:
            with lock:
                if (state["next"] >= len(work) or time.perf_counter() - t0 >= budget_s
                        or (max_rows and state["next"] >= max_rows)):
                    return
                b, qb = work[state["next"]]
                state["next"] += 1
            lo = cu[b] + qb * pb.block_size_q
            hi = min(lo + pb.block_size_q, cu[b + 1])
            o.prefill_topk(pb.q_idx[lo:hi], pb.k_idx_cache, pb.block_table, pb.slot_ids[b:b + 1],
                           torch.tensor([0, hi - lo], dtype=torch.int32), pb.seq_lens[b:b + 1],
                           torch.tensor([pre[b] + qb * pb.block_size_q], dtype=torch.int32),
                           torch.tensor([0, 1], dtype=torch.int32), pb.block_size_q, pb.init_blocks,
                           pb.local_blocks, float(np.float32(pb.scale)), 1, pb.topk)
            with lock:
                state["done"] += hi - lo

    pool = [threading.Thread(target=worker) for _ in range(max(1, threads))]
    for th in pool:
        th.start()
    for th in pool:
        th.join()
    dt = time.perf_counter() - t0
    return state["done"] / dt, state["done"], dt


def prefill_desc(pb):
    return {"workload": W.PREFILL_BATCH_NAME, "sequences": pb.B, "query_tokens": int(pb.q_idx.shape[0]),
            "query_blocks": pb.n_rows, "block_size_q": pb.block_size_q, "init_blocks": pb.init_blocks,
            "local_blocks": pb.local_blocks, "top_k": pb.topk, "index_heads": pb.Hi, "index_dim": pb.Di,
            "page_table_blocks": pb.NB, "pool_pages": pb.P, "prefix_lens": pb.prefix_lens.tolist(),
            "index_dtype": str(pb.q_idx.dtype)[6:],
            "l2": "flushed between timed steps (256 MiB rewrite, then a 256 MiB read that cleans the dirty "
                  "lines; outside the events)"}


def run_prefill_reference(args, rank, world):
    if rank != 0:
        return None
    pb = W.prefill_batch()
    cores = host_cores()
    per_step_budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        prefill_oracle_rate(pb, budget_s=per_step_budget / 4, max_rows=1)
    rows, secs = 0, 0.0
    for _ in range(args.steps):
        _, n, dt = prefill_oracle_rate(pb, budget_s=per_step_budget, threads=cores)
        rows += n
        secs += dt
    value = rows / secs
    return {
        "impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": prefill_desc(pb),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": "%d query tokens (whole query blocks) through the oracle (single-threaded "
                                   "C, fp64, called from %d host threads), %.1f s per step"
                                   % (rows, cores, per_step_budget)},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_prefill_gpu(args, rank, world, local_rank):
    import sparse_paged_decode_gb300 as spd

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pb = W.prefill_batch(seed=1004 + 97 * rank)
    g = pb.to(dev)
    total_q = int(pb.q_idx.shape[0])
    out = torch.empty((pb.Hi, pb.n_rows, pb.topk), dtype=torch.int32, device=dev)
    ws = torch.empty(spd.prefill_workspace_bytes(total_q, pb.Hi, pb.NB), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    clean = torch.ones(FLUSH_BYTES // 4, dtype=torch.int32, device=dev)
    clean_sum = torch.empty((), dtype=torch.int64, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        torch.sum(clean, 0, dtype=torch.int64, out=clean_sum)

    def step():
        spd.msa_prefill_block_score(g.q_idx, g.k_idx_cache, g.block_table, g.slot_ids, g.cu_seqlens, g.seq_lens,
                                    g.prefix_lens, pb.block_size_q, BS, pb.init_blocks, pb.local_blocks, pb.scale,
                                    g.cu_seqblocks_q, out, ws)

    for i in range(args.warmup):
        flush_l2(i)
        step()
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.25)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    n0 = spd.launch_count()
    for i in range(args.steps):
        flush_l2(i)
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize(dev)
    launches = spd.launch_count() - n0
    if world > 1:
        torch.distributed.barrier()
    step_ms = [a.elapsed_time(b) for a, b in evs]

    # end to end: the batch's index queries and metadata copied in from
    # pinned host memory (the index cache stays resident), the ids copied back
    per_call = [("q_idx", pb.q_idx), ("slot_ids", pb.slot_ids), ("cu_seqlens", pb.cu_seqlens),
                ("seq_lens", pb.seq_lens), ("prefix_lens", pb.prefix_lens), ("cu_seqblocks_q", pb.cu_seqblocks_q)]
    hosts = [(getattr(g, k), t.contiguous().pin_memory()) for k, t in per_call]
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(h.numel() * h.element_size() for _, h in hosts)
    d2h = host_out.numel() * host_out.element_size()
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush_l2(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for d, h in hosts:
            d.copy_(h, non_blocking=True)
        step()
        host_out.copy_(out, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    clocks = sampler.stop() if sampler else None

    total_ms, e2e_total = max_over_ranks([sum(step_ms), sum(e2e_ms)], world, dev)
    if rank != 0:
        return None
    value = job_rate(total_q, world, args.steps, total_ms)
    e2e_value = job_rate(total_q, world, args.steps, e2e_total)
    flops = prefill_flops(pb)
    mean_s = statistics.mean(step_ms) / 1e3
    achieved = flops / mean_s / 1e12
    peak, peak_src = measured_bf16_peak()
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline_record(lambda b, n: prefill_oracle_rate(pb, budget_s=b, threads=n),
                                  "query tokens (whole query blocks) of the batch", args.cpu_seconds)
    return {
        "metric": PREFILL_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 mma, f32 accumulate", "data": "synthetic",
        "config": prefill_desc(pb),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": None,
                     "kernel": "fused prefill call (token limits, score_tc_kernel, selection; direct launch)",
                     "algorithmic_flops_per_launch": flops, "mean_launch_us": mean_s * 1e6,
                     "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "timed_as": "direct launches per step",
        "clocks": clocks,
        "step_ms_median": statistics.median(step_ms),
    }


def _kernel_stamp(kv_cache="e4m3"):
    try:
        from sparse_paged_decode_gb300 import build as b

        return b._stamp(b.ATTENTION_SOURCES[kv_cache])[:16]
    except Exception:  # pragma: no cover
        return None


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=lambda c: c if c in ("dense", "prefill") else int(c), default=5,
                    choices=[2, 3, 4, 5, "dense", "prefill"],
                    help="workload (5 = stress sparse decode, the headline; 2 = EAGLE-style verification "
                         "decode; 3 = dense paged decode; 4 = batched prefill score-to-selection; "
                         "dense = the dense-attention prefill chunk; prefill = the fused prefill "
                         "score-to-selection call)")
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch each call directly instead of replaying a graph")
    ap.add_argument("--index-cache", default="native", choices=["native", "e4m3"],
                    help="index cache as generated (bf16) or stored FP8-E4M3")
    ap.add_argument("--kv-cache", default="e4m3", choices=["e4m3", "bf16"],
                    help="K/V cache as FP8-E4M3 with static scalar scales (default) or dense BF16")
    ap.add_argument("--attention-kernel", default="auto", choices=["auto", "general", "lanes", "rows"],
                    help="paged attention kernel: the tensor-core kernel of the cache type (default), the "
                         "general-layout kernel, or for an FP8 cache the keys-on-lanes or the query-rows "
                         "tensor-core kernel")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    ref_arm = {"dense": run_dense_reference, "prefill": run_prefill_reference}.get(args.config, run_reference)
    gpu_arm = {"dense": run_dense_gpu, "prefill": run_prefill_gpu}.get(args.config, run_gpu)
    if args.impl == "reference":
        # the oracle arm runs on rank 0 only; other ranks exit without work
        res = ref_arm(args, rank, world)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend="nccl")
    try:
        res = gpu_arm(args, rank, world, local_rank)
    except TimedOutWait as e:
        print("bench: %s" % e, file=sys.stderr, flush=True)
        sys.exit(3)
    if res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

"""Benchmark: paged GQA decode attention on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--repeats R] [--workload NAME] [--impl pkv|reference]
    python bench.py --trace-study [--calibrate]

Default workload: batch-1 long context (1 x 32768 tokens, 32 query / 8 KV heads,
D 128, 16-token pages scattered over a 4096-page pool, 32 splits).  One step is
one pkv_decode: the split-partial kernel over the compact queue with the LSE
merge fused into its last-arriving splits.  Metric: KV-read GB/s (KV bytes of
the step / device time of the step) and µs per step; roofline fraction against
the measured HBM copy bandwidth.  The same JSON line also carries, under
"workloads", the mixed batch (8 rows, log-uniform lengths), the high batch
(64 x 4096) and the continuous sessions (56 sessions, 200 steps of append +
re-plan + decode, p50 / p99), each gated on the fp64 oracle first and sampled
for clocks on its own (--headline-only leaves them out).

Timing rules: parity against the fp64 oracle before any timing; W >= 3 warm-up
steps; clocks sampled with nvidia-smi during the timed region.  The timed
region is K steps back to back between one pair of CUDA events on the
launching stream, repeated R times; the line gives the median per-step time of
the R regions and their min and max.  Inputs are cold: R copies of the page
pool and q are used round robin, with R chosen so that at least 6 x L2 bytes
are read between two reads of the same copy (a step that is itself over 6 x L2
needs no copy).  Steps too small for that (the tiny case) are timed one by one
after an L2 flush (a 2 x L2-size buffer written).  Each step is also timed
alone, after a flush, between its own events ("isolated_us_per_step"), which
adds the launch latency to every step.  Multi-GPU (torchrun, one rank per GPU)
runs independent replicas of the workload, partitioned by sequence: no
collective on the data path, a barrier and max-over-ranks timing only.

--workload trace:<kind>:<B> times one batch of a PersistentKV trace family
(uniform, bimodal, zipf, bucketed) on the policy's route.  --trace-study runs
every family at B = 1, 4, 8 on every route (each batch parity-gated), with the
summary's scheduler counters; --calibrate first fits the policy thresholds on
the calibration seed.

--impl reference times the fp64 CPU oracle on the host cores on the same
workload and metric (a bounded sample per step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/step and KV-read GB/s (fraction of GB300 HBM peak)"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
PROFILE_DIR = os.path.join(ROOT, "profiles")
KERNEL_SOURCE = os.path.join(ROOT, "paged_kv_decode_block_gb300", "csrc", "pkv_attention.cu")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(values, dist, device):
    """Element-wise maximum of a list of floats over all ranks (the slowest rank
    sets the time of a multi-GPU step); returns the list unchanged on one rank."""
    if dist is None or not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    with open(KERNEL_SOURCE, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(PROFILE_DIR, f"attention_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_src = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]{16})", text)
    m_bytes = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    if not m_src or not m_bytes or m_src.group(1) != kernel_source_hash():
        return None
    return int(m_bytes.group(1))


def smi_index(local: int) -> int:
    """nvidia-smi index of this rank's GPU (CUDA_VISIBLE_DEVICES may remap it)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [x.strip() for x in vis.split(",") if x.strip()]
    if local < len(parts) and parts[local].isdigit():
        return int(parts[local])
    return local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workloads

WORKLOAD_NAMES = ("batch1_long", "mixed", "mixed_padded", "high_batch", "tiny", "continuous")


def parse_trace_name(name: str):
    """'trace:<kind>:<B>' -> (kind, B); None for the named workloads."""
    from paged_kv_decode_block_gb300 import workloads as wl
    if not name.startswith("trace:"):
        return None
    parts = name.split(":")
    if len(parts) != 3 or parts[1] not in wl.TRACE_KINDS or not parts[2].isdigit() or int(parts[2]) < 1:
        raise ValueError(f"bad trace workload {name!r}: want trace:<{'|'.join(wl.TRACE_KINDS)}>:<batch>")
    return parts[1], int(parts[2])


def build_workload(name: str, seed: int | None = None):
    from paged_kv_decode_block_gb300 import workloads as wl
    tr = parse_trace_name(name)
    if tr is not None:   # a trace-family batch on the policy's own route
        return wl.trace(tr[0], tr[1], wl.HELD_OUT_SEED if seed is None else seed), dict()
    makers = {"batch1_long": (wl.batch1_long, dict(force_mode="split_queue", num_splits=32)),
              "mixed": (wl.mixed, dict(force_mode="split_queue")),
              "mixed_padded": (wl.mixed, dict(force_mode="split_padded")),
              "high_batch": (wl.high_batch, dict()),
              "tiny": (wl.tiny, dict(force_mode="split_queue", num_splits=4)),
              "continuous": (wl.continuous, dict(force_mode="persistent", num_splits=1))}
    make, opts = makers[name]
    return (make() if seed is None else make(seed)), opts


def workload_config(p, name: str, world: int = 1) -> dict:
    """The workload part of the JSON line's config, shared by both arms."""
    return {"workload": p.name, "batch": p.B,
            "seq_lens": "32768" if name == "batch1_long" else f"sum {int(p.seq_lens.sum())}",
            "q_heads": p.Hq, "kv_heads": p.Hkv, "head_dim": p.D, "page_size": p.page_size,
            "num_pages": p.num_pages, "requested_splits": int(p.num_splits),
            "parallelism": f"replicas x{world} (partition by sequence, no collective)"}


def parity_gate(p, out, lse, nthreads):
    import oracle
    ref_out, ref_lse = oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, nthreads=nthreads)
    err_out = float(np.max(np.abs(out - ref_out)))
    fin = np.isfinite(ref_lse)
    err_lse = float(np.max(np.abs(lse[fin] - ref_lse[fin]))) if fin.any() else 0.0
    ok = err_out <= 2e-3 and err_lse <= 1e-4 and np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    return ok, err_out, err_lse


# what one attention launch does on each route, for the roofline line
ROUTE_WORDS = {
    "split_queue": "split partials over the compact queue, LSE merge fused",
    "split_padded": "split partials over the padded split grid, LSE merge fused",
    "direct": "one tile per (row, KV head), finalised in place",
    "persistent": "persistent CTAs draining the queue, LSE merge fused",
}


def route_words(info: dict) -> str:
    words = ROUTE_WORDS.get(info["mode_name"], info["mode_name"])
    if info["merge_name"] == "separate":
        return words.replace("LSE merge fused", "LSE merge in its own launch")
    if info["merge_name"] == "none":
        return words.replace(", LSE merge fused", "")
    return words


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(p, budget_s: float, nthreads: int):
    """Run full oracle steps until `budget_s` has passed (at least one); seconds per step."""
    import oracle
    oracle.load()
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, nthreads=nthreads)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return (time.perf_counter() - t0) / n, n


def single_thread_oracle(p, kv_bytes: int, estimate_s: float, limit_s: float = 15.0):
    """One full oracle step on one thread, when it should take under `limit_s`
    (estimated from the threaded step); else None."""
    if estimate_s > limit_s:
        return None
    sec, _ = time_oracle(p, 0.0, 1)
    return {"value": round(kv_bytes / sec / 1e9, 4), "unit": "GB/s", "cores": 1, "ms_per_step": round(sec * 1e3, 1)}


# ----------------------------------------------------------------------------- our arm

def phase_summary(rows, pkv):
    """Median phase durations (µs) of one traced attention launch, from its
    per-CTA timeline rows (pkv_trace_read)."""
    t = rows.astype(np.int64)
    ran = t[:, pkv.TR_TILES] > 0
    streamed = ran & (t[:, pkv.TR_FIRST_BLOCK] > 0)
    t0 = int(t[:, pkv.TR_WAIT_DONE].min())

    def med(a, b, sel):
        v = (t[sel, b] - t[sel, a]) / 1e3
        return round(float(np.median(v)), 3) if v.size else None

    merged = t[:, pkv.TR_MERGE_END] > 0
    arrived = t[:, pkv.TR_ARRIVED] > 0
    out = {"ctas": int(len(t)), "ctas_with_tiles": int(ran.sum()),
           "wait_released_spread": round(float((t[:, pkv.TR_WAIT_DONE].max() - t0) / 1e3), 3),
           "wait_to_first_block": med(pkv.TR_WAIT_DONE, pkv.TR_FIRST_BLOCK, streamed),
           "stream": med(pkv.TR_FIRST_BLOCK, pkv.TR_STREAM_END, streamed),
           "combine": med(pkv.TR_STREAM_END, pkv.TR_COMBINE_END, ran),
           "arrival": med(pkv.TR_COMBINE_END, pkv.TR_ARRIVED, ran & arrived),
           "merge": med(pkv.TR_ARRIVED, pkv.TR_MERGE_END, merged),
           "stream_end_median_to_last": round(float((t[streamed, pkv.TR_STREAM_END].max()
                                                     - np.median(t[streamed, pkv.TR_STREAM_END])) / 1e3), 3)
           if streamed.any() else None,
           "launch_span": round(float((t[:, pkv.TR_EXIT].max() - t0) / 1e3), 3)}
    if merged.any():
        out["last_merge_end"] = round(float((t[merged, pkv.TR_MERGE_END].max() - t0) / 1e3), 3)
    return out

def device_problem(p, dev):
    """The problem's inputs in device memory, plus fp32 outputs."""
    import torch
    return dict(q=torch.from_numpy(p.q.view(np.int16)).to(dev),
                k=torch.from_numpy(p.k_pages.view(np.int16)).to(dev),
                v=torch.from_numpy(p.v_pages.view(np.int16)).to(dev),
                table=torch.from_numpy(p.block_table).to(dev),
                lens=torch.from_numpy(p.seq_lens).to(dev),
                out=torch.empty((p.B, p.Hq, p.D), dtype=torch.float32, device=dev),
                lse=torch.empty((p.B, p.Hq), dtype=torch.float32, device=dev))


def decode_line(name, args, ctx, headline=True):
    """Parity-gate, then time, pkv_decode on one workload; returns its JSON dict.
    headline=False gives the compact form carried inside the headline line's
    `workloads` object (no e2e, no CPU baseline, no isolated per-kernel split)."""
    import torch
    from paged_kv_decode_block_gb300 import pkv

    dist, dev, world, rank, local = ctx["dist"], ctx["dev"], ctx["world"], ctx["rank"], ctx["local"]
    p, opts = build_workload(name)
    opts = dict(opts, math=args.math, separate_merge=args.separate_merge, copy=args.copy, merge=args.merge)
    if headline and args.num_splits is not None:
        opts["num_splits"] = args.num_splits
    if headline and args.mode is not None:
        opts["force_mode"] = args.mode
    d = device_problem(p, dev)
    q, k, v, table, lens, out, lse = (d[x] for x in ("q", "k", "v", "table", "lens", "out", "lse"))
    plan = pkv.Plan(p.seq_lens, p.block_table, p.page_size, B=p.B, Hq=p.Hq, Hkv=p.Hkv, D=p.D,
                    max_pages=p.max_pages, num_pages=p.num_pages, **opts)
    info = plan.info()
    stream = torch.cuda.current_stream()

    # correctness gate before any timing
    pkv.decode(q, k, v, table, lens, plan, out, lse)
    torch.cuda.synchronize()
    if plan.status() != 0:
        raise SystemExit(f"{name}: device status word set on the parity run")
    ok, err_out, err_lse = parity_gate(p, out.cpu().numpy(), lse.cpu().numpy(), host_cores())
    log(f"{name}: parity vs oracle: max|out|={err_out:.3g} max|lse|={err_lse:.3g} -> {'ok' if ok else 'FAIL'}")
    if not ok:
        raise SystemExit(f"{name}: parity gate failed; not timing")

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    step_bytes = info["kv_bytes"] + p.B * p.Hq * p.D * 2
    # Cold inputs without a flush: R copies of the page pool (and q), used round
    # robin, so that at least 6 x L2 bytes are read between two reads of a copy
    # (the L2 keeps a few percent of lines across 3 x L2 of streaming, measured
    # with ncu; across 6 x L2 under 0.3 %).
    rot = 1 if step_bytes >= 6 * l2 else 1 + -(-6 * l2 // step_bytes)
    if args.copies:
        rot = args.copies   # e.g. 1 under a profiler, which flushes caches itself
    streamed = rot <= 16
    copies = [(q, k, v)] + [(q.clone(), k.clone(), v.clone()) for _ in range(rot - 1 if streamed else 0)]
    # The clones leave their last pages in L2 at normal priority, where the
    # kernel's evict-first loads would never displace them: flush once.
    flush.zero_()
    n_launch = info["launches_per_step"]
    per_kernel_events = n_launch > 1

    def step(i):
        qi, ki, vi = copies[i % len(copies)]
        pkv.decode(qi, ki, vi, table, lens, plan, out, lse)

    for i in range(args.warmup):
        if not streamed:
            flush.zero_()
        step(i)
    torch.cuda.synchronize()

    # (1) the timed region, repeated: K steps back to back on cold copies between
    # one event pair (or, when the step is too small for that, with an L2 flush
    # before every step, each step between its own events)
    K, R = args.steps, args.repeats
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(R)]
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    region_ms = []
    with ClockSampler(smi_index(local)) as clk:
        time.sleep(0.3)
        # a soak of the same steps right before the timed region, so that the
        # 200 ms clock samples see the GPU under this load
        t_soak = time.perf_counter()
        i = 0
        while time.perf_counter() - t_soak < args.soak:
            for _ in range(100):
                step(i)
                i += 1
            torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t_wall0 = time.perf_counter()
        for r in range(R):
            if streamed:
                ev[r][0].record(stream)
                for i in range(K):
                    step(r * K + i)
                ev[r][1].record(stream)
            else:
                for i in range(K):
                    flush.zero_()
                    starts[i].record(stream)
                    step(i)
                    ends[i].record(stream)
                torch.cuda.synchronize()
                region_ms.append(statistics.median(s.elapsed_time(e) for s, e in zip(starts, ends)))
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t_wall = time.perf_counter() - t_wall0
        time.sleep(0.3)
    if streamed:
        region_ms = [a.elapsed_time(b) / K for a, b in ev]
    med_ms = statistics.median(region_ms)

    # (2) for reference: every step alone, between its own events (adds the
    # launch latency to each step), after one of two L2 flushes: writing a
    # 2 x L2 buffer (the L2 is then full of dirty lines, whose write-back to HBM
    # lands inside the timed kernel as it evicts them), or reading a 2 x L2
    # buffer that is never written (the L2 then holds clean lines of another
    # buffer, and the previous step's dirty lines were written back during the
    # sweep); per-kernel events when the step has two launches
    clean = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.int32, device=dev)
    plan.profile(per_kernel_events)
    iso_ms, iso_clean_ms, kernel_ms = [], [], []
    for i in range(max(min(K, 50), 5)):
        for dirty, acc in ((True, iso_ms), (False, iso_clean_ms)):
            if dirty:
                flush.zero_()
            else:
                clean.sum()
            starts[i % K].record(stream)
            step(i)
            ends[i % K].record(stream)
            ends[i % K].synchronize()
            acc.append(starts[i % K].elapsed_time(ends[i % K]))
            if per_kernel_events and dirty:
                kernel_ms.append(plan.profile_read())
            elif per_kernel_events:
                plan.profile_read()
    plan.profile(False)
    del clean
    iso_med = statistics.median(iso_ms)
    iso_clean_med = statistics.median(iso_clean_ms)
    if per_kernel_events:
        attn_ms = statistics.mean(km[0] for km in kernel_ms)
        merge_ms = statistics.mean(km[1] for km in kernel_ms)
    else:
        attn_ms = med_ms
        merge_ms = 0.0

    med_ms, attn_ms, iso_med, iso_clean_med, lo_ms, hi_ms = reduce_max(
        [med_ms, attn_ms, iso_med, iso_clean_med, min(region_ms), max(region_ms)], dist, dev)
    kv = info["kv_bytes"]
    q_bytes = p.B * p.Hq * p.D * 2
    o_bytes = p.B * p.Hq * (p.D + 1) * 4
    alg_bytes_attn = kv + q_bytes   # what the attention kernel must read
    value = kv * world / (med_ms * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    achieved = alg_bytes_attn / (attn_ms * 1e-3) / 1e9
    clocks = clk.summary()
    clocks = {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"],
              "samples": clocks["samples"]}
    us = {"median": round(med_ms * 1e3, 2), "min": round(lo_ms * 1e3, 2), "max": round(hi_ms * 1e3, 2),
          "repeats": R, "steps_per_repeat": K}
    l2_words = (f"cold: {rot} cop{'y' if rot == 1 else 'ies'} of the page pool and q used round robin, >= 6 x L2 bytes read between "
                f"two reads of a copy; {R} repeats of {K} steps back to back, one event pair each"
                if streamed else f"flushed before every timed step (2 x L2 bytes written); {R} repeats of "
                                 f"{K} steps, median step of each")
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_src,
                "kernel": f"attention_kernel ({route_words(info)})",
                "algorithmic_bytes_per_launch": alg_bytes_attn, "traffic": profiled_traffic(name)}
    if not headline:
        return {"workload": p.name, "mode": info["mode_name"], "merge": info["merge_name"],
                "tiles": info["num_work_items"], "chunk_pages": info["chunk_pages"],
                "kv_bytes_per_step": kv, "us_per_step": us, "isolated_us_per_step": round(iso_med * 1e3, 2),
                "isolated_clean_l2_us_per_step": round(iso_clean_med * 1e3, 2),
                "kv_gbs": round(value, 2), "frac_of_measured": round(value / peak, 4),
                "frac_of_nominal_7_9TBs": round(value / NOMINAL_HBM_GBS, 4), "roofline": roofline,
                "l2": l2_words, "clocks": clocks,
                "parity": {"max_abs_out": err_out, "max_abs_lse": err_lse}}

    phases = None
    if args.phase_trace:
        # per-CTA timelines of the last step of a back-to-back run, repeated
        plan.trace(True)
        runs = []
        for r in range(R):
            for i in range(K):
                step(i)
            runs.append(phase_summary(plan.read_trace(), pkv))
        plan.trace(False)
        phases = {k: (round(statistics.median(x[k] for x in runs), 3) if isinstance(runs[0][k], float) else runs[0][k])
                  for k in runs[0] if all(r.get(k) is not None for r in runs)}
        phases["note"] = (f"median over {R} traced launches (each the last of {K} back-to-back steps) of per-CTA "
                          "median phase durations in us; times from the grid dependency wait's release")

    # end to end through the C ABI with host buffers: host re-plan, then
    # pkv_decode_host, which synchronises: the kernel reads the new plan and q in
    # pinned host memory and writes out + lse there (over NVLink-C2C, no copy
    # engine); wall time per step, each step cold (L2 flushed before it)
    q_host = torch.from_numpy(p.q.view(np.int16)).pin_memory()
    out_host = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    lse_host = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    e2e_s, replan_s, call_s = [], [], []
    for i in range(args.warmup + K):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        plan.update(p.seq_lens)
        t1 = time.perf_counter()
        pkv.decode_host(q_host, k, v, table, lens, plan, out_host, lse_host)
        if i >= args.warmup:
            t2 = time.perf_counter()
            e2e_s.append(t2 - t0)
            replan_s.append(t1 - t0)
            call_s.append(t2 - t1)
    e2e_med = statistics.median(e2e_s)
    # the same call's kernel alone, device time between events after the same flush
    dev_ms = []
    for i in range(max(min(K, 20), 5)):
        plan.update(p.seq_lens)
        flush.zero_()
        starts[i % K].record(stream)
        pkv.decode_host(q_host, k, v, table, lens, plan, out_host, lse_host)
        ends[i % K].record(stream)
        ends[i % K].synchronize()
        dev_ms.append(starts[i % K].elapsed_time(ends[i % K]))
    breakdown = {"replan_us": round(statistics.median(replan_s) * 1e6, 2),
                 "decode_host_call_us": round(statistics.median(call_s) * 1e6, 2),
                 "device_us": round(statistics.median(dev_ms) * 1e3, 2)}
    breakdown["host_and_sync_us"] = round(breakdown["decode_host_call_us"] - breakdown["device_us"], 2)
    if not (np.array_equal(out_host.numpy(), out.cpu().numpy()) and np.array_equal(lse_host.numpy(), lse.cpu().numpy())):
        raise SystemExit("the host-buffer path disagrees with the device path")
    upload = 4 * (5 * info["num_work_items"] + 2 * p.B) if info["mode"] != pkv.MODE_DIRECT else 0
    e2e_med = reduce_max([e2e_med], dist, dev)[0]

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu:
        cores = host_cores()
        sec, n = time_oracle(p, args.cpu_budget, cores)
        cpu = {"value": round(kv / sec / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} full oracle decode step(s) of the same workload (fp64 C, {cores} threads), "
                         f"{sec * 1e3:.0f} ms per step"}
        cpu["single_thread"] = single_thread_oracle(p, kv, sec * cores)

    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(med_ms, 5),
        "us_per_step": round(med_ms * 1e3, 2), "us_per_step_spread": us,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16 in, fp32 accumulate", "data": "synthetic (seeded, bf16 ~N(0,1))",
        "config": {**workload_config(p, name, world),
                   "mode": info["mode_name"], "math": args.math, "copy": info["copy_name"],
                   "merge": info["merge_name"],
                   "num_splits": info["max_splits"],
                   "chunk_pages": info["chunk_pages"], "tiles": info["num_work_items"],
                   "empty_tiles": info["empty_tiles"], "merge_state_bytes": info["workspace_bytes"],
                   "launches_per_step": info["launches_per_step"], "l2": l2_words},
        "kv_bytes_per_step": kv,
        "isolated_us_per_step": round(iso_med * 1e3, 2),
        "isolated_clean_l2_us_per_step": round(iso_clean_med * 1e3, 2),
        "isolated_note": ("each step alone between its own events, launch latency included, after an L2 flush: "
                          "isolated_us_per_step after writing 2 x L2 (its dirty lines are written back inside "
                          "the timed kernel), isolated_clean_l2_us_per_step after reading 2 x L2 of a buffer "
                          "never written (clean lines)"),
        "frac_of_nominal_7_9TBs": round(value / NOMINAL_HBM_GBS, 4),
        "kernel_ms": {"attention": round(attn_ms, 5), "merge": round(merge_ms, 5)},
        "roofline": roofline,
        "e2e": {"value": round(kv * world / e2e_med / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e_med * 1e6, 2), "h2d_bytes_per_step": q_bytes + upload,
                "d2h_bytes_per_step": o_bytes,
                "path": "host re-plan + pkv_decode_host: the kernel reads the plan and q from pinned host "
                        "memory and writes out/lse to pinned host memory (NVLink-C2C), then a synchronise",
                "breakdown": {**breakdown,
                              "note": "medians per step: the host re-plan; the pkv_decode_host call (launch, "
                                      "kernel, synchronise); the kernel's device time between events on the "
                                      "stream after the same L2 flush (launch latency included); the call "
                                      "minus that device time (host launch work and the wake-up of the "
                                      "synchronise)"}},
        "gpu_launches": n_launch * K * R,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "timed_region_wall_s": round(t_wall, 4),
        "parity": {"max_abs_out": err_out, "max_abs_lse": err_lse},
        **({"phases_us": phases} if phases else {}),
    }


def dist_context(args):
    import torch
    import torch.distributed as dist
    rank, world, local = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    return {"dist": dist, "dev": torch.device("cuda", local), "world": world, "rank": rank, "local": local}


def release_memory():
    import gc
    import torch
    gc.collect()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


# the other workloads the headline line carries (each parity-gated, with its own clocks)
SIDE_WORKLOADS = ("mixed", "high_batch", "continuous")


def run_pkv(args):
    from paged_kv_decode_block_gb300 import pkv

    ctx = dist_context(args)
    pkv.load()
    line = decode_line(args.workload, args, ctx)
    if args.workload == "batch1_long" and not args.headline_only:
        side = {}
        for name in SIDE_WORKLOADS:
            release_memory()
            if name == "continuous":
                side[name] = continuous_line(args, ctx, steps=200, warmup=max(args.warmup, 5), headline=False)
            else:
                side[name] = decode_line(name, args, ctx, headline=False)
        line["workloads"] = side
        line["gpu_launches"] += sum(w.get("gpu_launches", 0) for w in side.values())
        for w in side.values():
            w.pop("gpu_launches", None)
    if ctx["rank"] == 0:
        print(json.dumps(line), flush=True)
    if ctx["world"] > 1:
        ctx["dist"].destroy_process_group()


# ----------------------------------------------------------------------------- continuous sessions

def continuous_line(args, ctx, steps=None, warmup=None, headline=True):
    """56 sessions; every step appends one K/V token per session (a fresh page from
    the pool when one fills), re-plans on the host and decodes with the persistent
    queue kernel.  Device time per step covers append + host re-plan + decode (the
    GPU waits while the host plans, as a serving loop would); wall time adds the
    host-side pool work and a synchronise.  Each step reads ~1 GB of KV, far more
    than L2, so no flush is needed between steps."""
    import torch
    from paged_kv_decode_block_gb300 import pkv
    from paged_kv_decode_block_gb300 import workloads as wl
    from paged_kv_decode_block_gb300.session import ContinuousSessions

    local = ctx["local"]
    steps = args.steps if steps is None else steps
    warmup = args.warmup if warmup is None else warmup
    total = warmup + steps
    e2e_steps = min(8, steps)
    p = wl.continuous(steps=total + e2e_steps + 1)   # room for every appended token (e2e and profiling steps too)
    splits = 1 if (args.num_splits is None or not headline) else args.num_splits
    device_plan = headline and (args.device_plan or args.graph)
    use_graph = headline and args.graph
    sess = ContinuousSessions(p, force_mode="persistent", num_splits=splits, math=args.math, copy=args.copy)
    rng = np.random.default_rng(wl.HELD_OUT_SEED + 1)
    toks = [wl.new_tokens(rng, p.B, p.Hkv, p.D) for _ in range(total)]
    k_new = torch.from_numpy(np.stack([t[0] for t in toks]).view(np.int16)).cuda()
    v_new = torch.from_numpy(np.stack([t[1] for t in toks]).view(np.int16)).cuda()
    stream = torch.cuda.current_stream()

    # correctness gate on the first step
    sess.step(k_new[0], v_new[0])
    torch.cuda.synchronize()
    if sess.plan.status() != 0:
        raise SystemExit("continuous: device status word set on the parity step")
    import oracle
    table0 = sess.table_h.copy()
    k0, v0, lens0 = oracle.append(toks[0][0], toks[0][1], p.k_pages, p.v_pages, table0, p.seq_lens)
    ref_out, ref_lse = oracle.decode(p.q, k0, v0, table0, lens0, nthreads=host_cores())
    del k0, v0
    err_out = float(np.max(np.abs(sess.out.cpu().numpy() - ref_out)))
    err_lse = float(np.max(np.abs(sess.lse.cpu().numpy() - ref_lse)))
    log(f"continuous: parity vs oracle (step 0): max|out|={err_out:.3g} max|lse|={err_lse:.3g}")
    if err_out > 2e-3 or err_lse > 1e-4:
        raise SystemExit("continuous: parity gate failed; not timing")

    if device_plan:
        sess.session.device_plan()
    kbuf = torch.empty_like(k_new[0])
    vbuf = torch.empty_like(v_new[0])
    graph = None

    def one_step(i):
        if graph is None:
            sess.step(k_new[i], v_new[i])
        else:   # the captured step reads its tokens from fixed buffers
            kbuf.copy_(k_new[i])
            vbuf.copy_(v_new[i])
            graph.replay()

    for i in range(1, warmup):
        one_step(i)
    torch.cuda.synchronize()
    if use_graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                sess.step(kbuf, vbuf)
        stream.wait_stream(side)
        # capturing enqueued nothing; the lengths still match the host's count
    lens0 = sess.lens_h.astype(np.int64).sum()
    sess.plan.profile(not use_graph)
    dev_us, wall_us, kv, attn_ms = [], [], [], []
    with ClockSampler(smi_index(local)) as clk:
        time.sleep(0.3)
        torch.cuda.synchronize()
        t_region = time.perf_counter()
        for n, i in enumerate(range(warmup, total)):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            a.record(stream)
            one_step(i)
            b.record(stream)
            b.synchronize()
            wall_us.append((time.perf_counter() - t0) * 1e6)
            dev_us.append(a.elapsed_time(b) * 1e3)
            if not use_graph:
                attn_ms.append(sess.plan.profile_read()[0])
            kv.append(int(lens0 + (n + 1) * p.B) * p.Hkv * p.D * 4)
        t_region = time.perf_counter() - t_region
        time.sleep(0.3)
    sess.plan.profile(False)
    if use_graph:   # kernel time of the attention launch, from one more profiled eager step
        sess.plan.profile(True)
        torch.cuda.synchronize()
        sess.step(k_new[total - 1], v_new[total - 1])
        attn_ms = [sess.plan.profile_read()[0]] * len(kv)
        sess.plan.profile(False)
    kv_total = float(np.sum(kv))
    value = kv_total / (np.sum(dev_us) * 1e-6) / 1e9
    peak, peak_src = hbm_peak()
    q_bytes = p.B * p.Hq * p.D * 2
    achieved = float(np.mean([(k + q_bytes) / (t * 1e-3) / 1e9 for k, t in zip(kv, attn_ms)]))
    clocks = clk.summary()
    clocks = {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"], "reasons": clocks["reasons"],
              "samples": clocks["samples"]}
    p50, p99 = float(np.percentile(dev_us, 50)), float(np.percentile(dev_us, 99))
    info = sess.plan.info()
    launches = 1 + info["launches_per_step"] + (1 if device_plan else 0)
    roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": peak_src,
                "kernel": "attention_kernel (persistent queue drain)",
                "algorithmic_bytes_per_launch": int(np.mean(kv)) + q_bytes,
                "traffic": profiled_traffic("continuous")}
    step_words = ("CUDA-graph replay of device plan + append + persistent decode" if use_graph else
                  "device plan + append + persistent decode" if device_plan else
                  "append + host re-plan + persistent decode")
    if not headline:
        return {"workload": p.name, "mode": info["mode_name"], "sessions": p.B, "steps": steps,
                "step": step_words, "tiles": info["num_work_items"], "kv_bytes_per_step": int(np.mean(kv)),
                "us_per_step": {"device_p50": round(p50, 2), "device_p99": round(p99, 2),
                                "wall_p50": round(float(np.percentile(wall_us, 50)), 2),
                                "wall_p99": round(float(np.percentile(wall_us, 99)), 2),
                                "decode_kernel_mean": round(float(np.mean(attn_ms)) * 1e3, 2)},
                "decode_frac_of_measured": round(achieved / peak, 4),
                "step_frac_of_measured": round(float(np.mean(kv)) / (p50 * 1e-6) / 1e9 / peak, 4),
                "roofline": roofline, "clocks": clocks, "gpu_launches": launches * steps,
                "parity": {"max_abs_out": err_out, "max_abs_lse": err_lse, "checked_step": 0}}

    # end to end: new tokens and q from pinned host memory each step, outputs back to the host
    kh = torch.from_numpy(np.stack([t[0] for t in toks[:8]]).view(np.int16)).pin_memory()
    vh = torch.from_numpy(np.stack([t[1] for t in toks[:8]]).view(np.int16)).pin_memory()
    qh = torch.from_numpy(p.q.view(np.int16)).pin_memory()
    oh = torch.empty(sess.out.shape, dtype=torch.float32).pin_memory()
    lh = torch.empty(sess.lse.shape, dtype=torch.float32).pin_memory()
    kd, vd = torch.empty_like(k_new[0]), torch.empty_like(v_new[0])
    e2e = []
    for i in range(e2e_steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        kd.copy_(kh[i], non_blocking=True)
        vd.copy_(vh[i], non_blocking=True)
        sess.q.copy_(qh, non_blocking=True)
        sess.step(kd, vd)
        oh.copy_(sess.out, non_blocking=True)
        lh.copy_(sess.lse, non_blocking=True)
        torch.cuda.synchronize()
        e2e.append(time.perf_counter() - t0)
    e2e_med = statistics.median(e2e)

    return {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": ctx["world"], "steps": steps,
        "warmup": warmup, "ms_per_step": round(p50 / 1e3, 5),
        "us_per_step": {"device_p50": round(p50, 2), "device_p99": round(p99, 2),
                        "wall_p50": round(float(np.percentile(wall_us, 50)), 2),
                        "wall_p99": round(float(np.percentile(wall_us, 99)), 2)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 accumulate", "data": "synthetic (seeded, bf16 ~N(0,1))",
        "config": {"workload": p.name, "sessions": p.B, "seq_lens": "U[1024, 8192] + appended",
                   "q_heads": p.Hq, "kv_heads": p.Hkv, "head_dim": p.D, "page_size": p.page_size,
                   "num_pages": p.num_pages, "mode": info["mode_name"], "math": args.math, "copy": info["copy_name"],
                   "num_splits": info["max_splits"], "tiles": info["num_work_items"],
                   "grid_ctas": info["grid_ctas"], "launches_per_step": launches,
                   "l2": "not flushed: each step reads ~1 GB of KV, far above L2", "step": step_words},
        "kv_bytes_per_step": int(np.mean(kv)),
        "kernel_ms": {"attention_mean": round(float(np.mean(attn_ms)), 5)},
        "roofline": roofline,
        "e2e": {"value": round(float(np.mean(kv)) / e2e_med / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(e2e_med * 1e6, 2),
                "h2d_bytes_per_step": 2 * p.B * p.Hkv * p.D * 2 + q_bytes,
                "d2h_bytes_per_step": p.B * p.Hq * (p.D + 1) * 4},
        "gpu_launches": launches * steps,
        "cpu_baseline": None,
        "clocks": clocks,
        "timed_region_wall_s": round(t_region, 4),
        "parity": {"max_abs_out": err_out, "max_abs_lse": err_lse, "checked_step": 0},
    }


def run_continuous(args):
    from paged_kv_decode_block_gb300 import pkv
    ctx = dist_context(args)
    pkv.load()
    line = continuous_line(args, ctx)
    if ctx["rank"] == 0:
        print(json.dumps(line), flush=True)


def run_resident(args):
    """The continuous-session workload on one resident kernel (pkv_resident_*):
    launched once, it runs every step the host publishes (device plan, append,
    persistent decode, grid barriers between them).  Each step's new tokens and
    q go host -> device from pinned memory, and out / lse come back, inside the
    step call.  Device time per step comes from the kernel's own globaltimer
    stamps (step seen -> outputs published); the decode phase's stamps give the
    attention time for the roofline."""
    import torch
    import oracle
    from paged_kv_decode_block_gb300 import pkv
    from paged_kv_decode_block_gb300 import workloads as wl
    from paged_kv_decode_block_gb300.session import ContinuousSessions

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    pkv.load()
    steps = args.steps
    total = args.warmup + steps
    p = wl.continuous(steps=total + 1)
    splits = 1 if args.num_splits is None else args.num_splits
    sess = ContinuousSessions(p, force_mode="persistent", num_splits=splits, math=args.math, copy=args.copy)
    sess.session.device_plan()
    rng = np.random.default_rng(wl.HELD_OUT_SEED + 1)
    toks = [wl.new_tokens(rng, p.B, p.Hkv, p.D) for _ in range(total)]
    kh = torch.from_numpy(np.stack([t[0] for t in toks]).view(np.int16)).pin_memory()
    vh = torch.from_numpy(np.stack([t[1] for t in toks]).view(np.int16)).pin_memory()
    qh = torch.from_numpy(p.q.view(np.int16)).pin_memory()
    oh = torch.empty(sess.out.shape, dtype=torch.float32).pin_memory()
    lh = torch.empty(sess.lse.shape, dtype=torch.float32).pin_memory()
    kbuf = torch.empty((p.B, p.Hkv, p.D), dtype=torch.int16, device="cuda")
    vbuf = torch.empty_like(kbuf)
    lens0 = int(p.seq_lens.astype(np.int64).sum())
    torch.cuda.synchronize()
    res = pkv.Resident(sess.session, sess.k, sess.v, sess.q, kbuf, vbuf, sess.out, sess.lse,
                       idle_limit_ns=20_000_000_000, times_cap=total)
    wall_us = []
    try:
        # correctness gate on the first step (the kernel waits while the host checks)
        res.step(q_h=qh, k_new_h=kh[0], v_new_h=vh[0], out_h=oh, lse_h=lh)
        table0 = p.block_table.copy()
        free = list(p.free_pages)
        for b in range(p.B):
            if p.seq_lens[b] % p.page_size == 0 and table0[b, p.seq_lens[b] // p.page_size] < 0:
                table0[b, p.seq_lens[b] // p.page_size] = free.pop(0)
        k0, v0, l0 = oracle.append(toks[0][0], toks[0][1], p.k_pages, p.v_pages, table0, p.seq_lens)
        ref_out, ref_lse = oracle.decode(p.q, k0, v0, table0, l0, nthreads=host_cores())
        del k0, v0
        err_out = float(np.max(np.abs(oh.numpy() - ref_out)))
        err_lse = float(np.max(np.abs(lh.numpy() - ref_lse)))
        log(f"parity vs oracle (step 0): max|out|={err_out:.3g} max|lse|={err_lse:.3g}")
        if err_out > 2e-3 or err_lse > 1e-4:
            raise SystemExit("parity gate failed; not timing")
        for i in range(1, args.warmup):
            res.step(q_h=qh, k_new_h=kh[i], v_new_h=vh[i], out_h=oh, lse_h=lh)
        with ClockSampler(smi_index(local)) as clk:
            time.sleep(0.3)
            t_region = time.perf_counter()
            for i in range(args.warmup, total):
                t0 = time.perf_counter()
                res.step(q_h=qh, k_new_h=kh[i], v_new_h=vh[i], out_h=oh, lse_h=lh)
                wall_us.append((time.perf_counter() - t0) * 1e6)
            t_region = time.perf_counter() - t_region
            time.sleep(0.3)
    finally:
        res.stop()
    stamps = res.times().astype(np.int64)[args.warmup:total]
    res.close()
    if sess.plan.status() != 0:
        raise SystemExit("device status word set")
    dev_us = (stamps[:, 3] - stamps[:, 0]) / 1e3
    dec_us = (stamps[:, 3] - stamps[:, 2]) / 1e3
    plan_us = (stamps[:, 1] - stamps[:, 0]) / 1e3     # slot requests, allocation and plan, grid barrier
    append_us = (stamps[:, 2] - stamps[:, 1]) / 1e3   # CTA 0's appends until its drain starts
    kv = [(lens0 + (i + 1) * p.B) * p.Hkv * p.D * 4 for i in range(args.warmup, total)]
    value = float(np.sum(kv)) / (float(np.sum(dev_us)) * 1e-6) / 1e9
    peak, peak_src = hbm_peak()
    q_bytes = p.B * p.Hq * p.D * 2
    achieved = float(np.mean([(k + q_bytes) / (t * 1e-6) / 1e9 for k, t in zip(kv, dec_us)]))
    clocks = clk.summary()
    info = sess.plan.info()
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(float(np.median(dev_us)) / 1e3, 5),
        "us_per_step": {"device_p50": round(float(np.percentile(dev_us, 50)), 2),
                        "device_p99": round(float(np.percentile(dev_us, 99)), 2),
                        "plan_phase_p50": round(float(np.percentile(plan_us, 50)), 2),
                        "append_phase_p50": round(float(np.percentile(append_us, 50)), 2),
                        "decode_phase_p50": round(float(np.percentile(dec_us, 50)), 2),
                        "wall_p50": round(float(np.percentile(wall_us, 50)), 2),
                        "wall_p99": round(float(np.percentile(wall_us, 99)), 2)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 in, fp32 accumulate", "data": "synthetic (seeded, bf16 ~N(0,1))",
        "config": {"workload": p.name, "sessions": p.B, "seq_lens": "U[1024, 8192] + appended",
                   "q_heads": p.Hq, "kv_heads": p.Hkv, "head_dim": p.D, "page_size": p.page_size,
                   "num_pages": p.num_pages, "mode": "resident (one cooperative launch for all steps)",
                   "math": args.math, "copy": info["copy_name"], "num_splits": splits,
                   "l2": "not flushed: each step reads ~1 GB of KV, far above L2",
                   "step": "device plan + append + persistent decode inside one resident kernel, grid barriers "
                           "between them; the host publishes each step through mapped pinned memory"},
        "kv_bytes_per_step": int(np.mean(kv)),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "kernel": "resident_kernel, decode phase (append done -> outputs published)",
                     "algorithmic_bytes_per_launch": int(np.mean(kv)) + q_bytes, "traffic": None},
        "e2e": {"value": round(float(np.mean(kv)) / (float(np.median(wall_us)) * 1e-6) / 1e9, 2), "unit": "GB/s",
                "us_per_step": round(float(np.median(wall_us)), 2),
                "h2d_bytes_per_step": 2 * p.B * p.Hkv * p.D * 2 + q_bytes,
                "d2h_bytes_per_step": p.B * p.Hq * (p.D + 1) * 4},
        "gpu_launches": 1,
        "cpu_baseline": None,
        "clocks": {"sm_mhz": clocks["sm_mhz"], "sm_max_mhz": clocks["sm_max_mhz"],
                   "reasons": clocks["reasons"], "samples": clocks["samples"]},
        "timed_region_wall_s": round(t_region, 4),
        "parity": {"max_abs_out": err_out, "max_abs_lse": err_lse, "checked_step": 0},
        "tiles": info["num_work_items"],
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- trace-family study

STUDY_ROUTES = ("auto", "split_queue", "split_padded", "direct", "persistent")
STUDY_BATCHES = (1, 4, 8)


def _study_time_route(p, dev, route, policy, steps, flush):
    """Median device µs of one pkv_decode on `route`, each step alone after an L2 flush."""
    import torch
    from paged_kv_decode_block_gb300 import pkv
    opts = dict(policy)
    if route != "auto":
        opts["force_mode"] = route
    plan = pkv.Plan(p.seq_lens, p.block_table, p.page_size, B=p.B, Hq=p.Hq, Hkv=p.Hkv, D=p.D,
                    max_pages=p.max_pages, num_pages=p.num_pages, **opts)
    stream = torch.cuda.current_stream()
    for _ in range(3):
        flush.zero_()
        pkv.decode(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], plan, dev["out"], dev["lse"])
    ts = []
    for _ in range(steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        pkv.decode(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], plan, dev["out"], dev["lse"])
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    if plan.status() != 0:
        raise SystemExit(f"device status set ({p.name}, {route})")
    info = plan.info()
    plan.close()
    return statistics.median(ts), info


def _study_parity(p, dev, policy):
    """The policy route against the oracle (exits on a mismatch)."""
    from paged_kv_decode_block_gb300 import pkv
    plan = pkv.Plan(p.seq_lens, p.block_table, p.page_size, B=p.B, Hq=p.Hq, Hkv=p.Hkv, D=p.D,
                    max_pages=p.max_pages, num_pages=p.num_pages, **policy)
    pkv.decode(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], plan, dev["out"], dev["lse"])
    ok, err_out, err_lse = parity_gate(p, dev["out"].cpu().numpy(), dev["lse"].cpu().numpy(), host_cores())
    plan.close()
    if not ok:
        raise SystemExit(f"parity failed on {p.name}: {err_out}, {err_lse}")
    return err_out, err_lse


def trace_study(seed, policy, steps, dev, routes=STUDY_ROUTES, batches=STUDY_BATCHES, emit=print):
    """Every trace family at every batch size: parity of the policy route, then the
    step time of every route, with the PersistentKV summary's scheduler counters
    (launches per step against 2 per distinct length for exact-length buckets,
    tiles, empty tiles of the padded grid, merge-state bytes)."""
    import torch
    from paged_kv_decode_block_gb300 import workloads as wl
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    rows = []
    for kind in wl.TRACE_KINDS:
        for B in batches:
            p = wl.trace(kind, B, seed)
            d = device_problem(p, dev)
            errs = _study_parity(p, d, policy)
            kv = p.kv_bytes()
            for route in routes:
                us, info = _study_time_route(p, d, route, policy, steps, flush)
                row = dict(seed=seed, trace=kind, batch=B, route=route, mode=info["mode_name"],
                           us_per_step=round(us, 2), kv_gbs=round(kv / (us * 1e-6) / 1e9, 1),
                           launches=info["launches_per_step"],
                           exact_bucket_launches=2 * len(set(int(n) for n in p.seq_lens)),
                           tiles=info["num_work_items"], empty_tiles=info["empty_tiles"],
                           chunk_pages=info["chunk_pages"], merge_state_bytes=info["workspace_bytes"],
                           kv_bytes=kv, lens=[int(n) for n in p.seq_lens], parity_out=errs[0],
                           parity_lse=errs[1])
                rows.append(row)
                emit(json.dumps(row))
            del d
            release_memory()
    return rows


def calibrate_policy(seed, steps, dev, emit=print):
    """Pick (target_ctas_per_sm, min_chunk_pages) minimising the geometric mean of the
    policy route's step time over every trace family and batch size at `seed` (the
    summary's calibration seed; thresholds fitted on one seed, reported on the other)."""
    import itertools
    import math
    import torch
    from paged_kv_decode_block_gb300 import workloads as wl
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    grid = list(itertools.product((1, 2, 3, 4), (4, 8, 16, 32)))
    scores = {g: [] for g in grid}
    for kind in wl.TRACE_KINDS:
        for B in STUDY_BATCHES:
            p = wl.trace(kind, B, seed)
            d = device_problem(p, dev)
            for tc, mc in grid:
                us, _ = _study_time_route(p, d, "auto", dict(target_ctas_per_sm=tc, min_chunk_pages=mc), steps,
                                          flush)
                scores[(tc, mc)].append(us)
            del d
            release_memory()
    geo = {g: math.exp(statistics.mean(math.log(x) for x in v)) for g, v in scores.items()}
    for g in sorted(geo, key=geo.get):
        emit(json.dumps(dict(seed=seed, target_ctas_per_sm=g[0], min_chunk_pages=g[1], geomean_us=round(geo[g], 2))))
    best = min(geo, key=geo.get)
    return dict(target_ctas_per_sm=best[0], min_chunk_pages=best[1])


def run_trace_study(args):
    """--trace-study [--calibrate]: one JSON row per (trace, batch, route) on stdout."""
    from paged_kv_decode_block_gb300 import pkv
    from paged_kv_decode_block_gb300 import workloads as wl
    ctx = dist_context(args)
    if ctx["rank"] != 0:
        return
    pkv.load()
    policy = {}
    if args.calibrate:
        policy = calibrate_policy(wl.CALIBRATION_SEED, args.study_steps, ctx["dev"])
        print(json.dumps({"calibration": policy, "seed": wl.CALIBRATION_SEED}), flush=True)
    trace_study(wl.HELD_OUT_SEED, policy, args.study_steps, ctx["dev"])


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    p, _ = build_workload(args.workload)
    kv = p.kv_bytes()
    cores = host_cores()
    budget = args.cpu_budget / max(1, args.steps)   # each step: at least one full oracle decode
    for _ in range(args.warmup):
        time_oracle(p, 0.0, cores)
    per_step = []
    for _ in range(args.steps):
        sec, _n = time_oracle(p, budget, cores)
        per_step.append(sec)
    sec = statistics.median(per_step)
    value = kv / sec / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, bf16 ~N(0,1))",
        "config": {**workload_config(p, args.workload, world), "mode": "fp64 CPU oracle (host cores)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step = full oracle decode of the workload, repeated for ~{budget:.1f} s"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--repeats", type=int, default=5,
                    help="timed regions of --steps steps each; the line reports their median, min and max")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed steps before each timed region")
    ap.add_argument("--workload", default="batch1_long",
                    help=f"one of {', '.join(WORKLOAD_NAMES)}, or trace:<kind>:<batch>")
    ap.add_argument("--headline-only", action="store_true",
                    help="batch1_long: leave out the other workloads the line otherwise carries")
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--math", default="auto", choices=["auto", "fma", "mma"],
                    help="block reduction: tensor cores (mma.sync) or CUDA-core FMA")
    ap.add_argument("--separate-merge", action="store_true", help="merge splits in a second launch")
    ap.add_argument("--merge", default="auto", choices=["auto", "last", "all"],
                    help="fused merge: the last arriving split, or every split sharing out the outputs")
    ap.add_argument("--mode", default=None, choices=["auto", "direct", "split_queue", "split_padded", "persistent"],
                    help="override the workload's route")
    ap.add_argument("--num-splits", type=int, default=None,
                    help="override the workload's split count (0 = the planner's policy)")
    ap.add_argument("--copy", default="auto", choices=["auto", "lsu", "tma"],
                    help="K/V staging: cp.async from the producer warp, or TMA boxes")
    ap.add_argument("--device-plan", action="store_true",
                    help="continuous: plan each step on the device (pkv_session_device_plan)")
    ap.add_argument("--graph", action="store_true",
                    help="continuous: device-planned step captured once in a CUDA graph and replayed")
    ap.add_argument("--resident", action="store_true",
                    help="continuous workload: one resident kernel runs every step (pkv_resident_*)")
    ap.add_argument("--copies", type=int, default=0,
                    help="copies of the inputs used round robin (default: enough for >= 6 x L2 between reuses)")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for the CPU baseline")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--trace-study", action="store_true",
                    help="every trace family x batch 1/4/8 x route, parity-gated; one JSON row each")
    ap.add_argument("--calibrate", action="store_true",
                    help="with --trace-study: fit the policy thresholds on the calibration seed first")
    ap.add_argument("--study-steps", type=int, default=15, help="timed steps per route in the trace study")
    ap.add_argument("--phase-trace", action="store_true",
                    help="add the per-CTA phase timeline (pkv_trace_*) of back-to-back steps to the line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.repeats < 1 or args.steps < 1:
        ap.error("--repeats and --steps must be >= 1")
    if args.workload not in WORKLOAD_NAMES:
        try:
            if parse_trace_name(args.workload) is None:
                raise ValueError(f"unknown workload {args.workload!r}")
        except ValueError as e:
            ap.error(str(e))
    if args.impl == "reference":
        run_reference(args)
    elif args.trace_study:
        run_trace_study(args)
    elif args.workload == "continuous" and args.resident:
        run_resident(args)
    elif args.workload == "continuous":
        run_continuous(args)
    else:
        run_pkv(args)


if __name__ == "__main__":
    main()

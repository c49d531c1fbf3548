"""Trace-family study and policy calibration.

    python -m paged_kv_decode_block_gb300.tracestudy [--calibrate] [--steps 20] [--out FILE]

Reproduces, on one GB300, the evaluation shape of "PersistentKV: Page-Aware
Decode Scheduling for Long-Context LLM Serving on Commodity GPUs"
(gist.science summary), Methodology section 3 and Results:
  * the four trace families (Uniform, Bimodal, Zipf-like, Bucketed; see
    workloads.trace) at batch sizes 1, 4 and 8;
  * every route of the planner (compact queue, padded split grid, direct
    single-pass, persistent queue) next to the policy's own choice;
  * the summary's scheduler counters: launches per step (and, for reference,
    the 2 launches per distinct length that exact-length buckets would need),
    tiles, empty tiles of the padded grid, and merge-state bytes;
  * thresholds calibrated on the calibration seed 20260622 and reported on the
    held-out seed 20260623 ("Results": fixed thresholds from one seed, numbers
    on the other).
Every batch is first checked against the fp64 oracle.  Device time per step is
taken with CUDA events around pkv_decode, median of --steps, with L2 flushed
before each step.
"""
from __future__ import annotations

import argparse
import itertools
import json
import math
import statistics
import sys

import numpy as np
import torch

from . import pkv
from . import workloads as wl

ROUTES = ("auto", "split_queue", "split_padded", "direct", "persistent")
BATCHES = (1, 4, 8)


def _device(p):
    return dict(q=torch.from_numpy(p.q.view(np.int16)).cuda(),
                k=torch.from_numpy(p.k_pages.view(np.int16)).cuda(),
                v=torch.from_numpy(p.v_pages.view(np.int16)).cuda(),
                table=torch.from_numpy(p.block_table).cuda(),
                lens=torch.from_numpy(p.seq_lens).cuda(),
                out=torch.empty((p.B, p.Hq, p.D), dtype=torch.float32, device="cuda"),
                lse=torch.empty((p.B, p.Hq), dtype=torch.float32, device="cuda"))


def _plan(p, route, policy):
    opts = dict(policy)
    if route != "auto":
        opts["force_mode"] = route
    return pkv.Plan(p.seq_lens, p.block_table, p.page_size, B=p.B, Hq=p.Hq, Hkv=p.Hkv, D=p.D,
                    max_pages=p.max_pages, num_pages=p.num_pages, **opts)


def time_route(p, dev, route, policy, steps, flush):
    plan = _plan(p, route, policy)
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
        raise RuntimeError(f"device status set ({route})")
    return statistics.median(ts), plan.info()


def parity(p, dev, policy):
    """Policy route against the oracle (raises on a mismatch)."""
    import oracle   # the tests' fp64 definition; only this check uses it
    plan = _plan(p, "auto", policy)
    pkv.decode(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], plan, dev["out"], dev["lse"])
    ref_out, ref_lse = oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, nthreads=16)
    err_out = float(np.max(np.abs(dev["out"].cpu().numpy() - ref_out)))
    err_lse = float(np.max(np.abs(dev["lse"].cpu().numpy() - ref_lse)))
    if err_out > 2e-3 or err_lse > 1e-4:
        raise RuntimeError(f"parity failed on {p.name}: {err_out}, {err_lse}")
    return err_out, err_lse


def study(seed, policy, steps, routes=ROUTES, kinds=wl.TRACE_KINDS, batches=BATCHES, check=True, log=print):
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    rows = []
    for kind, B in itertools.product(kinds, batches):
        p = wl.trace(kind, B, seed)
        dev = _device(p)
        errs = parity(p, dev, policy) if check else (None, None)
        kv = p.kv_bytes()
        for route in routes:
            us, info = time_route(p, dev, route, policy, steps, flush)
            row = dict(seed=seed, trace=kind, batch=B, route=route, mode=info["mode_name"], us_per_step=round(us, 2),
                       kv_gbs=round(kv / (us * 1e-6) / 1e9, 1), launches=info["launches_per_step"],
                       exact_bucket_launches=2 * len(set(int(n) for n in p.seq_lens)),
                       tiles=info["num_work_items"], empty_tiles=info["empty_tiles"],
                       chunk_pages=info["chunk_pages"], merge_state_bytes=info["workspace_bytes"],
                       kv_bytes=kv, lens=[int(n) for n in p.seq_lens], parity_out=errs[0], parity_lse=errs[1])
            rows.append(row)
            log(json.dumps(row))
        del dev
        torch.cuda.empty_cache()
    return rows


def calibrate(seed, steps, log=print):
    """Pick (target_ctas_per_sm, min_chunk_pages) minimising the geometric mean of the
    policy route's step time over every trace and batch size at `seed`."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    grid = list(itertools.product((1, 2, 3, 4), (4, 8, 16, 32)))
    scores = {g: [] for g in grid}
    for kind, B in itertools.product(wl.TRACE_KINDS, BATCHES):
        p = wl.trace(kind, B, seed)
        dev = _device(p)
        for tc, mc in grid:
            us, _ = time_route(p, dev, "auto", dict(target_ctas_per_sm=tc, min_chunk_pages=mc), steps, flush)
            scores[(tc, mc)].append(us)
        del dev
        torch.cuda.empty_cache()
    geo = {g: math.exp(statistics.mean(math.log(x) for x in v)) for g, v in scores.items()}
    for g in sorted(geo, key=geo.get):
        log(json.dumps(dict(seed=seed, target_ctas_per_sm=g[0], min_chunk_pages=g[1], geomean_us=round(geo[g], 2))))
    best = min(geo, key=geo.get)
    return dict(target_ctas_per_sm=best[0], min_chunk_pages=best[1]), geo


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--calibrate", action="store_true", help="calibrate on 20260622, report on 20260623")
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--out", default=None, help="write all JSON rows to this file")
    args = ap.parse_args()
    pkv.load()
    rows = []
    policy = {}
    if args.calibrate:
        policy, geo = calibrate(wl.CALIBRATION_SEED, args.steps)
        rows.append(dict(calibration=policy, geomean_us={f"{k[0]},{k[1]}": round(v, 2) for k, v in geo.items()}))
        print(json.dumps(rows[-1]))
    rows += study(wl.HELD_OUT_SEED, policy, args.steps)
    if args.out:
        with open(args.out, "w") as f:
            for r in rows:
                f.write(json.dumps(r) + "\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())

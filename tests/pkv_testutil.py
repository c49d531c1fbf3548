"""Shared helpers for the GPU tests: move a seeded problem to the device, run
the CUDA path through the C ABI, and compare with the fp64 oracle.

Tolerances (max-abs, on identical seeded bf16 inputs): 2e-3 on the fp32
output, 1e-4 on the natural-log LSE.  Work queues must match the oracle's
enumeration bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_decode_block_gb300 import pkv
from paged_kv_decode_block_gb300 import workloads as wl

OUT_TOL = 2e-3
LSE_TOL = 1e-4


def to_device(p: wl.Problem, device="cuda"):
    return dict(
        q=torch.from_numpy(p.q.view(np.int16)).to(device),
        k=torch.from_numpy(p.k_pages.view(np.int16)).to(device),
        v=torch.from_numpy(p.v_pages.view(np.int16)).to(device),
        table=torch.from_numpy(p.block_table).to(device),
        lens=torch.from_numpy(p.seq_lens).to(device),
        out=torch.empty((p.B, p.Hq, p.D), dtype=torch.float32, device=device),
        lse=torch.empty((p.B, p.Hq), dtype=torch.float32, device=device),
    )


def make_plan(p: wl.Problem, host_table=True, **opts) -> pkv.Plan:
    return pkv.Plan(p.seq_lens, p.block_table if host_table else None, p.page_size, B=p.B, Hq=p.Hq,
                    Hkv=p.Hkv, D=p.D, max_pages=p.max_pages, num_pages=p.num_pages, **opts)


def run(p: wl.Problem, dev=None, plan=None, **opts):
    dev = dev or to_device(p)
    plan = plan or make_plan(p, **opts)
    pkv.decode(dev["q"], dev["k"], dev["v"], dev["table"], dev["lens"], plan, dev["out"], dev["lse"])
    torch.cuda.synchronize()
    return dev["out"].cpu().numpy(), dev["lse"].cpu().numpy(), plan, dev


def oracle_result(p: wl.Problem, nthreads: int = 8):
    return oracle.decode(p.q, p.k_pages, p.v_pages, p.block_table, p.seq_lens, nthreads=nthreads)


def assert_close(out, lse, ref_out, ref_lse, what=""):
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    err_out = np.max(np.abs(out - ref_out)) if out.size else 0.0
    assert err_out <= OUT_TOL, f"{what}: max |out - oracle| = {err_out:.3g} > {OUT_TOL}"
    neg = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), neg), f"{what}: -inf pattern of lse differs"
    if np.any(~neg):
        err_lse = np.max(np.abs(lse[~neg] - ref_lse[~neg]))
        assert err_lse <= LSE_TOL, f"{what}: max |lse - oracle| = {err_lse:.3g} > {LSE_TOL}"


def expected_queue(p: wl.Problem, plan_info: dict) -> np.ndarray:
    """The oracle's enumeration for the plan's chunk size and mode."""
    C = plan_info["chunk_pages"]
    mode = plan_info["mode"]
    if mode == pkv.MODE_SPLIT_PADDED:
        return oracle.enumerate_padded_grid(p.seq_lens, p.page_size, p.Hkv, C)
    if mode == pkv.MODE_DIRECT:
        return oracle.enumerate_direct(p.seq_lens, p.page_size, p.Hkv)
    return oracle.enumerate_queue(p.seq_lens, p.page_size, p.Hkv, C)

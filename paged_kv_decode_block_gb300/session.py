"""Continuous decode sessions: many rows that each grow by one token per step.

One step of the continuous-session workload ("WPK persistent kernel",
dotwave.ai: a fixed cohort of sessions advancing together; its page arenas are
fixed pools, "What has to exist instead"):
  1. host: the page pool hands a fresh page to every row whose next token starts
     a page (pkv_pool_reserve); the changed block table goes to the device;
  2. host: the plan is rebuilt for the lengths after the append
     (pkv_plan_update, same buffers, so device addresses stay fixed);
  3. device: pkv_append writes each row's new K/V token and bumps seq_lens;
  4. device: pkv_decode runs attention for every row.
This module only sequences those C-ABI calls and keeps the host mirrors of the
lengths and the table; all arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import pkv
from .workloads import Problem


class ContinuousSessions:
    def __init__(self, problem: Problem, device="cuda", **plan_opts):
        p = problem
        self.p = p
        self.page_size = p.page_size
        self.lens_h = p.seq_lens.astype(np.int32).copy()
        self.table_h = torch.from_numpy(p.block_table.copy()).pin_memory()   # host mirror, pinned
        self.q = torch.from_numpy(p.q.view(np.int16)).to(device)
        self.k = torch.from_numpy(p.k_pages.view(np.int16)).to(device)
        self.v = torch.from_numpy(p.v_pages.view(np.int16)).to(device)
        self.table_d = self.table_h.to(device)
        self.lens_d = torch.from_numpy(self.lens_h.copy()).to(device)
        self.out = torch.empty((p.B, p.Hq, p.D), dtype=torch.float32, device=device)
        self.lse = torch.empty((p.B, p.Hq), dtype=torch.float32, device=device)
        self.pool = pkv.Pool(p.free_pages if p.free_pages is not None else [], p.num_pages)
        self.plan = pkv.Plan(self.lens_h, None, p.page_size, B=p.B, Hq=p.Hq, Hkv=p.Hkv, D=p.D,
                             max_pages=p.max_pages, num_pages=p.num_pages, **plan_opts)
        self._table_copied = torch.cuda.Event()
        self._table_copied.record()
        torch.cuda.synchronize()

    def step(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor | None = None, stream=None):
        """Append one token per row, then decode.  k_new/v_new: device bf16 [B][Hkv][D]."""
        s = stream or torch.cuda.current_stream()
        self._table_copied.synchronize()          # the previous table upload has left the mirror
        rows = self.pool.reserve(self.lens_h, self.table_h.numpy(), self.page_size)
        if len(rows):
            with torch.cuda.stream(s):
                self.table_d.copy_(self.table_h, non_blocking=True)
                self._table_copied.record(s)
        # plan for the lengths after the append before launching anything, so that
        # append and decode reach the GPU back to back
        self.lens_h += 1
        self.plan.update(self.lens_h)
        pkv.append(k_new, v_new, self.k, self.v, self.table_d, self.lens_d, self.plan, stream=s)
        pkv.decode(self.q if q is None else q, self.k, self.v, self.table_d, self.lens_d, self.plan,
                   self.out, self.lse, stream=s)
        return len(rows)

    def kv_bytes(self) -> int:
        return int(self.lens_h.astype(np.int64).sum()) * self.p.Hkv * self.p.D * 2 * 2

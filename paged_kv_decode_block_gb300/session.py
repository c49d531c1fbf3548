"""Continuous decode sessions: many rows that each grow by one token per step.

One step of the continuous-session workload ("WPK persistent kernel",
dotwave.ai: a fixed cohort of sessions advancing together; its page arenas are
fixed pools, "What has to exist instead") is one native call, pkv_session_step:
  1. host: the page pool hands a fresh page to every row whose next token starts
     a page (pkv_pool_reserve);
  2. host: the plan is rebuilt for the lengths after the append
     (pkv_plan_update, same buffers, so device addresses stay fixed);
  3. device, one launch: the new table entries and the plan are read from
     pinned host memory and written to the device, and each row's new K/V
     token is appended (seq_lens += 1);
  4. device: pkv_decode runs attention for every row.
This module only owns the device tensors and forwards pointers; the sequencing
and all arithmetic run in the library.
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
        self.q = torch.from_numpy(p.q.view(np.int16)).to(device)
        self.k = torch.from_numpy(p.k_pages.view(np.int16)).to(device)
        self.v = torch.from_numpy(p.v_pages.view(np.int16)).to(device)
        self.table_d = torch.from_numpy(p.block_table.copy()).to(device)
        self.lens_d = torch.from_numpy(p.seq_lens.copy()).to(device)
        self.out = torch.empty((p.B, p.Hq, p.D), dtype=torch.float32, device=device)
        self.lse = torch.empty((p.B, p.Hq), dtype=torch.float32, device=device)
        self.pool = pkv.Pool(p.free_pages if p.free_pages is not None else [], p.num_pages)
        self.plan = pkv.Plan(p.seq_lens, None, p.page_size, B=p.B, Hq=p.Hq, Hkv=p.Hkv, D=p.D,
                             max_pages=p.max_pages, num_pages=p.num_pages, **plan_opts)
        torch.cuda.synchronize()
        self.session = pkv.Session(self.plan, self.pool, p.seq_lens, p.block_table, self.table_d, self.lens_d)

    def step(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor | None = None, stream=None):
        """Append one token per row, then decode.  k_new/v_new: device bf16 [B][Hkv][D]."""
        self.session.step(k_new, v_new, self.k, self.v, self.q if q is None else q, self.out, self.lse,
                          stream=stream)

    @property
    def lens_h(self) -> np.ndarray:
        return self.session.lengths()

    @property
    def table_h(self) -> np.ndarray:
        return self.session.table()

    def kv_bytes(self) -> int:
        return int(self.lens_h.astype(np.int64).sum()) * self.p.Hkv * self.p.D * 2 * 2

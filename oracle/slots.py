"""Continuous sessions with slot admit / evict -- oracle side.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Integer bookkeeping and
byte copies, checked bit for bit.

Sources:
  * "WPK persistent kernel" (dotwave.ai), "What has to exist instead": a fixed
    cohort of sessions advanced together, per-session state in fixed arenas whose
    slots are reset at a beat boundary;
  * "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving on
    Commodity GPUs" (gist.science summary), Methodology section 1 "Layout":
    token t of row b lives in page block_table[b][t // ps], slot t % ps.

Readings taken where the pages are silent (the rules the library implements):
  * one free list, first in first out; a step hands a page to every active row
    whose next token starts one, rows in order, before the append;
  * an eviction returns a row's pages (its non-negative table entries, in table
    order; rows in the order listed) to the back of the free list, sets its table
    entries to -1 and its length to 0, and makes the row idle: idle rows take no
    page and no token, and decode to the neutral state;
  * an admission gives an idle row ceil(n / ps) pages from the front of the free
    list (rows in the order listed, pages in table order), length n, and its
    prompt's n tokens of K and V written into those pages;
  * at one boundary, evictions come before admissions.
"""
from __future__ import annotations

from collections import deque

import numpy as np

from .append import append


def write_prompt(k_src, v_src, k_pages, v_pages, table_row, n_tokens: int):
    """Write tokens [0, n) of a prompt (k_src / v_src [n][Hkv][D]) into a row's pages, in place."""
    ps = k_pages.shape[1]
    for t in range(int(n_tokens)):
        page = int(table_row[t // ps])
        k_pages[page, t % ps] = k_src[t]
        v_pages[page, t % ps] = v_src[t]


class SlotModel:
    """The state of a session as the rules above change it: table, lengths, active
    flags, the free list, and (optionally) the K/V pools."""

    def __init__(self, seq_lens, block_table, free_pages, page_size: int, k_pages=None, v_pages=None):
        self.lens = np.array(seq_lens, dtype=np.int32, copy=True)
        self.table = np.array(block_table, dtype=np.int32, copy=True)
        self.free = deque(int(x) for x in free_pages)
        self.ps = int(page_size)
        self.active = np.ones(len(self.lens), dtype=np.int32)
        self.k_pages = k_pages
        self.v_pages = v_pages

    def evict(self, rows):
        for b in rows:
            assert self.active[b], f"row {b} is idle"
            for page in self.table[b]:
                if page >= 0:
                    self.free.append(int(page))
            self.table[b, :] = -1
            self.lens[b] = 0
            self.active[b] = 0

    def admit(self, rows, lens, k_src=None, v_src=None):
        """k_src / v_src: [sum(lens)][Hkv][D], the rows' tokens one after another."""
        at = 0
        for b, n in zip(rows, lens):
            assert not self.active[b], f"row {b} is active"
            need = -(-int(n) // self.ps)
            assert need <= len(self.free), "free list exhausted"
            for j in range(need):
                self.table[b, j] = self.free.popleft()
            self.lens[b] = int(n)
            self.active[b] = 1
            if self.k_pages is not None and n > 0:
                write_prompt(k_src[at:at + n], v_src[at:at + n], self.k_pages, self.v_pages, self.table[b], n)
            at += int(n)

    def step(self, k_new, v_new):
        """One step: pages for the active rows whose next token starts one, then the
        append of one token per active row (k_new / v_new [B][Hkv][D])."""
        for b in range(len(self.lens)):
            if not self.active[b] or self.lens[b] % self.ps != 0:
                continue
            idx = self.lens[b] // self.ps
            if self.table[b, idx] < 0:
                self.table[b, idx] = self.free.popleft()
        rows = np.nonzero(self.active)[0]
        if self.k_pages is not None and len(rows):
            lens = self.lens[rows].copy()
            append(k_new[rows], v_new[rows], self.k_pages, self.v_pages, self.table[rows], lens, inplace=True)
            self.lens[rows] = lens
        else:
            self.lens[rows] += 1

"""Work-tile enumeration for split-KV paged decode -- oracle side.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Written independently of
the planner in the product library; the two must agree bit for bit.

Source: "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM Serving
on Commodity GPUs" (gist.science summary), Technical Summary, Methodology
section 1: the sequence dimension is split into disjoint ranges ("Sequence
Splitting"); tile counts and split ranges come from each row's true length, and
empty splits do no KV reads ("Row-Local Bounds"); the compact work queue holds
only the non-empty (row, KV-head, split) intervals ("Compact Workqueue").

Readings taken where the page is silent:
  * split boundaries fall on page boundaries;
  * one chunk size C (in pages) per plan; row b has P_b = ceil(N_b / ps) pages
    and S_b = ceil(P_b / C) splits; split s covers pages [s*C, min((s+1)*C, P_b));
  * a requested split count S maps to C = ceil(P_max / S), P_max = max_b P_b;
  * queue order is lexicographic in (b, kvh, s);
  * the padded ("rectangular") grid has B * Hkv * S_max slots,
    S_max = ceil(P_max / C); slots with s >= S_b are empty;
  * the single-pass route (the summary's unsplit kernel for large batches,
    Methodology section 2) has one tile per (row, KV head) over the whole row,
    pages [0, P_b), split index 0, listed for every row in (b, kvh) order (an
    empty row's tile is empty and stands for its neutral state).
Each tile is the int32 record (b, kvh, s, page_begin, page_end), end exclusive.
"""
from __future__ import annotations

import numpy as np


def pages_of(n_tokens: int, page_size: int) -> int:
    """P_b: pages that hold n_tokens tokens."""
    return -(-int(n_tokens) // int(page_size))


def chunk_pages_for_splits(seq_lens, page_size: int, num_splits: int) -> int:
    """C = ceil(P_max / S); 1 when every row is empty."""
    p_max = max((pages_of(n, page_size) for n in seq_lens), default=0)
    if p_max == 0:
        return 1
    return -(-p_max // int(num_splits))


def enumerate_queue(seq_lens, page_size: int, num_kv_heads: int, chunk_pages: int) -> np.ndarray:
    """Compact queue: only the non-empty (b, kvh, s) tiles, lexicographic order."""
    tiles = []
    for b, n in enumerate(seq_lens):
        p_b = pages_of(n, page_size)
        s_b = -(-p_b // chunk_pages)
        for kvh in range(num_kv_heads):
            for s in range(s_b):
                tiles.append((b, kvh, s, s * chunk_pages, min((s + 1) * chunk_pages, p_b)))
    return np.array(tiles, dtype=np.int32).reshape(-1, 5)


def enumerate_padded_grid(seq_lens, page_size: int, num_kv_heads: int, chunk_pages: int) -> np.ndarray:
    """Rectangular grid of B * Hkv * S_max slots; empty slots have page_begin == page_end."""
    p = [pages_of(n, page_size) for n in seq_lens]
    s_max = -(-max(p, default=0) // chunk_pages)
    tiles = []
    for b, p_b in enumerate(p):
        for kvh in range(num_kv_heads):
            for s in range(s_max):
                begin = min(s * chunk_pages, p_b)
                end = min((s + 1) * chunk_pages, p_b)
                tiles.append((b, kvh, s, begin, end))
    return np.array(tiles, dtype=np.int32).reshape(-1, 5)


def enumerate_direct(seq_lens, page_size: int, num_kv_heads: int) -> np.ndarray:
    """Single-pass tiles: one per (b, kvh), the whole row, in (b, kvh) order."""
    tiles = []
    for b, n in enumerate(seq_lens):
        for kvh in range(num_kv_heads):
            tiles.append((b, kvh, 0, 0, pages_of(n, page_size)))
    return np.array(tiles, dtype=np.int32).reshape(-1, 5)

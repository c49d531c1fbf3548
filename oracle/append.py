"""KV-cache append of one token per (row, KV head) -- oracle side.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Byte work, checked bit
for bit.

Source: the paged layout of "PersistentKV: Page-Aware Decode Scheduling for
Long-Context LLM Serving on Commodity GPUs" (gist.science summary), Technical
Summary, Methodology section 1 "Layout": token t of row b lives in page
block_table[b][t // ps] at slot t % ps.  The KV-cache update operator of
"GPUOS" (arXiv 2604.17861, section 4, operator library) is the operation:
the new token of row b goes to position seq_lens[b], after which the length
grows by one.
"""
from __future__ import annotations

import numpy as np


def append(k_new, v_new, k_pages, v_pages, block_table, seq_lens, inplace=False):
    """Returns (k_pages, v_pages, seq_lens) after the append: updated copies, or the
    given arrays themselves updated in place when inplace=True (for long runs over
    large pools).

    k_new, v_new: [B][Hkv][D]; pages: [NP][ps][Hkv][D]; block_table [B][max_pages].
    Raises ValueError when a row has no room or its page id is out of range."""
    if not inplace:
        k_pages = np.array(k_pages, copy=True)
        v_pages = np.array(v_pages, copy=True)
        seq_lens = np.array(seq_lens, dtype=np.int32, copy=True)
    num_pages, page_size = k_pages.shape[0], k_pages.shape[1]
    for b in range(seq_lens.shape[0]):
        pos = int(seq_lens[b])
        logical = pos // page_size
        if logical >= block_table.shape[1]:
            raise ValueError(f"row {b} is full")
        page = int(block_table[b, logical])
        if not 0 <= page < num_pages:
            raise ValueError(f"row {b}: page id {page} out of range")
        slot = pos % page_size
        k_pages[page, slot] = k_new[b]
        v_pages[page, slot] = v_new[b]
        seq_lens[b] = pos + 1
    return k_pages, v_pages, seq_lens

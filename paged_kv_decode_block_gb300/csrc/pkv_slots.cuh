// pkv_slots.cuh -- slot admit / evict at a step boundary, as device functions
// (used by the slot kernels of pkv_append.cu and by the resident kernel of
// pkv_attention.cu).
//
// The rows of a continuous session are fixed slots, as the per-session state of
// "WPK persistent kernel" (dotwave.ai, "What has to exist instead") lives in
// fixed arenas whose slots are reset at a beat boundary.  An eviction returns a
// row's pages to the back of the free list and makes the row idle (length 0, no
// pages, skipped by the append and the page allocation); an admission takes a
// new session's pages from the front of the free list and copies its prompt's
// K/V into them, in the paged layout of "PersistentKV: Page-Aware Decode
// Scheduling for Long-Context LLM Serving on Commodity GPUs" (gist.science
// summary, Methodology section 1 "Layout": token t of row b in page
// block_table[b][t / page_size], slot t % page_size).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {
namespace slots {

// The bookkeeping of a batch of requests, by one thread: evictions first, then
// admissions, each in the order listed.  With a device free list (a ring of
// free_cap ids from index free_state[0], free_state[1] of them in use) the
// evicted pages go to its back and the admitted ones come from its front; an
// admission it cannot serve sets PKV_DEV_ROW_FULL and leaves that row and the
// ones after it idle.  With pages chosen on the host (free_list null) the table
// entries come from p.pages.
__device__ __forceinline__ void apply_requests(const SlotParams& p) {
    const int ps = p.page_size, mp = p.max_pages;
    uint32_t head = 0, avail = 0, cap = 0;
    if (p.free_list) {
        head = p.free_state[0];
        avail = p.free_state[1];
        cap = static_cast<uint32_t>(p.free_cap);
    }
    for (int i = 0; i < p.n; ++i) {
        const SlotRequest r = p.req[i];
        if (r.len >= 0 || r.row < 0 || r.row >= p.B) continue;
        int32_t* row = p.table + static_cast<size_t>(r.row) * mp;
        for (int j = 0; j < mp; ++j) {
            const int32_t page = row[j];
            if (page >= 0 && p.free_list) {
                if (page < p.num_pages && avail < cap) {
                    p.free_list[(head + avail) % cap] = page;
                    ++avail;
                } else {
                    atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_PAGE_OOB));
                }
            }
            row[j] = -1;
        }
        p.lens[r.row] = 0;
        p.active[r.row] = 0;
    }
    bool full = false;
    for (int i = 0; i < p.n; ++i) {
        const SlotRequest r = p.req[i];
        if (r.len < 0 || r.row < 0 || r.row >= p.B) continue;
        const int need = (r.len + ps - 1) / ps;
        int32_t* row = p.table + static_cast<size_t>(r.row) * mp;
        if (need > mp) full = true;
        if (p.free_list && static_cast<uint32_t>(need) > avail) full = true;
        if (full) {
            atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));
            continue;   // this row and every later admission stay idle
        }
        for (int j = 0; j < need; ++j) {
            if (p.free_list) {
                row[j] = p.free_list[head % cap];
                head = (head + 1) % cap;
                --avail;
            } else {
                row[j] = p.pages[r.page_off + j];
            }
        }
        p.lens[r.row] = r.len;
        p.active[r.row] = 1;
    }
    if (p.free_list) {
        p.free_state[0] = head;
        p.free_state[1] = avail;
    }
}

// Copy the prompts of the admitted rows (those the bookkeeping made active)
// into their pages: 16-byte vectors, the calling threads' share of a grid of
// `nthreads` threads numbered `tid`.
__device__ __forceinline__ void copy_prompts(const SlotParams& p, int64_t tid, int64_t nthreads) {
    const int row_elems = p.Hkv * p.D;   // one token of every KV head
    const int vecs = row_elems / 8;
    for (int i = 0; i < p.n; ++i) {
        const SlotRequest r = p.req[i];
        if (r.len <= 0 || r.row < 0 || r.row >= p.B || !p.active[r.row]) continue;
        const int32_t* table = p.table + static_cast<size_t>(r.row) * p.max_pages;
        const int64_t total = static_cast<int64_t>(r.len) * vecs;
        for (int64_t x = tid; x < total; x += nthreads) {
            const int t = static_cast<int>(x / vecs), c = static_cast<int>(x % vecs) * 8;
            const int page = table[t / p.page_size];
            if (page < 0 || page >= p.num_pages) continue;
            const size_t dst = (static_cast<size_t>(page) * p.page_size + t % p.page_size) * row_elems + c;
            const size_t src = (static_cast<size_t>(r.src_tok) + t) * row_elems + c;
            *reinterpret_cast<uint4*>(p.k_pages + dst) = *reinterpret_cast<const uint4*>(r.k_src + src);
            *reinterpret_cast<uint4*>(p.v_pages + dst) = *reinterpret_cast<const uint4*>(r.v_src + src);
        }
    }
}

}  // namespace slots
}  // namespace pkv

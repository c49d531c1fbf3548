// pkv_devplan.cuh -- the continuous-step planner, as a device function of one
// CTA (used by the planner kernel of pkv_devplan.cu and by the resident kernel
// of pkv_attention.cu).  See pkv_devplan.cu for the method and its citations.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {
namespace devplan {

// Exclusive prefix sum over the CTA of one int per thread (blockDim.x a
// multiple of 32, at most 1024); returns the thread's prefix and writes the
// total to *total.  `warp_sums`: 32 ints of shared memory.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* warp_sums) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    *total = warp_sums[nwarps - 1];
    __syncthreads();
    return before;
}

// Ints of shared scratch plan_step needs: four per-row arrays and 32 warp sums.
constexpr int kPlanScratchInts = 4 * kDevPlanMaxRows + 32;

// One planning step by the whole CTA of kThreads threads, on `scratch`
// (kPlanScratchInts ints of shared memory).  Rows go one per thread, in passes
// of kThreads rows, so a small batch still spreads over the CTA: each pass's
// prefix sums continue the last one's, which keeps everything in row order.
// The tiles are then written by all threads, each finding its tile's row by a
// binary search over the row starts.
template <int kThreads>
__device__ void plan_step(const DevPlanParams& p, int* scratch) {
    int* s_pages = scratch;                       // P_b after the append
    int* s_partial = s_pages + kDevPlanMaxRows;   // size of the row's last tile if partial, else 0
    int* s_start = s_partial + kDevPlanMaxRows;   // row_start
    int* s_full = s_start + kDevPlanMaxRows;      // hand-out slot of the row's first full-chunk tile
    int* warp_sums = s_full + kDevPlanMaxRows;    // 32
    const int tid = threadIdx.x;
    const int B = p.B, Hkv = p.Hkv, ps = p.page_size, C = p.chunk;
    if (B > kDevPlanMaxRows) {
        if (tid == 0) {
            atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
            *p.tiles = 0;
        }
        return;
    }
    const int passes = (B + kThreads - 1) / kThreads;

    // ---- 1. page allocation, in row order
    const uint32_t head = p.free_state[0], avail = p.free_state[1];
    int taken = 0;   // pages handed out by earlier passes
    for (int pass = 0; pass < passes; ++pass) {
        const int b = pass * kThreads + tid;
        int need = 0;
        if (b < B && (!p.active || p.active[b])) {   // idle slots take no page
            const int n = p.lens[b];
            if (n >= 0 && n % ps == 0) {
                if (n / ps >= p.max_pages)
                    atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));
                else if (p.table[static_cast<size_t>(b) * p.max_pages + n / ps] < 0)
                    need = 1;
            }
        }
        int total;
        const int rank = taken + block_exclusive_scan(need, &total, warp_sums);
        if (need) {
            if (static_cast<uint32_t>(rank) < avail) {
                const int n = p.lens[b];
                p.table[static_cast<size_t>(b) * p.max_pages + n / ps] =
                    p.free_list[(head + static_cast<uint32_t>(rank)) % static_cast<uint32_t>(p.free_cap)];
            } else {
                atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));   // pool exhausted
            }
        }
        taken += total;
    }
    if (tid == 0) {   // every thread read free_state before the first scan's barrier
        const uint32_t used = min(static_cast<uint32_t>(taken), avail);
        p.free_state[0] = (head + used) % static_cast<uint32_t>(p.free_cap);
        p.free_state[1] = avail - used;
    }

    // ---- 2. plan for the lengths after the append: splits, row starts, full-tile slots
    int total_tiles = 0, total_full = 0;
    for (int pass = 0; pass < passes; ++pass) {
        const int b = pass * kThreads + tid;
        int S = 0, F = 0;
        if (b < B) {
            const int n = max(p.lens[b], 0) + (!p.active || p.active[b] ? 1 : 0);   // idle slots do not grow
            const int pages = (n + ps - 1) / ps;
            S = (pages + C - 1) / C;
            const int rem = pages % C;
            F = rem == 0 ? S : S - 1;
            s_pages[b] = pages;
            s_partial[b] = rem;
        }
        int t_total, f_total;
        const int start = total_tiles + block_exclusive_scan(S * Hkv, &t_total, warp_sums);
        const int full_start = total_full + block_exclusive_scan(F * Hkv, &f_total, warp_sums);
        if (b < B) {
            s_start[b] = start;
            s_full[b] = full_start;
            p.row_start[b] = start;
            p.row_splits[b] = S;
        }
        total_tiles += t_total;
        total_full += f_total;
    }
    if (total_tiles > p.queue_cap) {
        if (tid == 0) {
            atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
            *p.tiles = 0;
        }
        return;
    }
    __syncthreads();   // the per-row arrays complete

    // ---- 3. the queue in (b, kvh, s) order, and the full-chunk tiles' hand-out slots
    for (int t = tid; t < total_tiles; t += kThreads) {
        int lo = 0, hi = B;   // first row whose tiles start after t
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (s_start[mid] <= t) lo = mid + 1;
            else hi = mid;
        }
        const int b = lo - 1;   // the last row starting at or before t: it holds t
        const int pages = s_pages[b];
        const int S = (pages + C - 1) / C;
        const int F = s_partial[b] == 0 ? S : S - 1;
        const int local = t - s_start[b];
        const int kvh = local / S, sp = local % S;
        p.queue[t] = pkv_work_item{b, kvh, sp, sp * C, min((sp + 1) * C, pages)};
        if (sp < F) p.order[s_full[b] + kvh * F + sp] = t;
    }

    // ---- 4. the partial tiles: rows ranked by their last tile's size (desc), then row
    for (int pass = 0; pass < passes; ++pass) {
        const int b = pass * kThreads + tid;
        if (b >= B || s_partial[b] == 0) continue;
        const int mine = s_partial[b];
        int before = 0;
        for (int c = 0; c < B; ++c) {
            const int other = s_partial[c];
            before += (other > mine) || (other == mine && c < b);
        }
        const int S = (s_pages[b] + C - 1) / C;
        const int row_start = s_start[b];
        for (int kvh = 0; kvh < Hkv; ++kvh)
            p.order[total_full + before * Hkv + kvh] = row_start + kvh * S + (S - 1);
    }
    if (tid == 0) *p.tiles = total_tiles;
}

}  // namespace devplan
}  // namespace pkv

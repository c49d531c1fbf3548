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

// One planning step by the whole CTA of kThreads threads.  Shared scratch:
// s_pages and s_partial of kDevPlanMaxRows ints each, warp_sums of 32 ints.
template <int kThreads>
__device__ void plan_step(const DevPlanParams& p, int* s_pages, int* s_partial, int* warp_sums) {
    constexpr int kRowsPerThread = (kDevPlanMaxRows + kThreads - 1) / kThreads;
    const int tid = threadIdx.x;
    const int B = p.B, Hkv = p.Hkv, ps = p.page_size, C = p.chunk;
    if (B > kDevPlanMaxRows) {
        if (tid == 0) {
            atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
            *p.tiles = 0;
        }
        return;
    }
    const int r0 = tid * kRowsPerThread;   // this thread's rows: [r0, r0 + kRowsPerThread)

    // ---- 1. page allocation, in row order
    int need[kRowsPerThread];
    int my_need = 0;
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        const int b = r0 + i;
        need[i] = 0;
        if (b < B && (!p.active || p.active[b])) {   // idle slots take no page
            const int n = p.lens[b];
            if (n >= 0 && n % ps == 0) {
                if (n / ps >= p.max_pages)
                    atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));
                else if (p.table[static_cast<size_t>(b) * p.max_pages + n / ps] < 0)
                    need[i] = 1;
            }
        }
        my_need += need[i];
    }
    int total_need;
    int rank = block_exclusive_scan(my_need, &total_need, warp_sums);
    const uint32_t head = p.free_state[0], avail = p.free_state[1];
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        if (!need[i]) continue;
        const int b = r0 + i;
        if (static_cast<uint32_t>(rank) < avail) {
            const int n = p.lens[b];
            p.table[static_cast<size_t>(b) * p.max_pages + n / ps] =
                p.free_list[(head + static_cast<uint32_t>(rank)) % static_cast<uint32_t>(p.free_cap)];
        } else {
            atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));   // pool exhausted
        }
        ++rank;
    }
    __syncthreads();
    if (tid == 0) {
        const uint32_t used = min(static_cast<uint32_t>(total_need), avail);
        p.free_state[0] = (head + used) % static_cast<uint32_t>(p.free_cap);
        p.free_state[1] = avail - used;
    }

    // ---- 2. plan for the lengths after the append
    int splits[kRowsPerThread], fulls[kRowsPerThread];
    int my_tiles = 0, my_full = 0;
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        const int b = r0 + i;
        splits[i] = fulls[i] = 0;
        if (b < B) {
            const int n = max(p.lens[b], 0) + (!p.active || p.active[b] ? 1 : 0);   // idle slots do not grow
            const int pages = (n + ps - 1) / ps;
            splits[i] = (pages + C - 1) / C;
            const int rem = pages % C;
            fulls[i] = rem == 0 ? splits[i] : splits[i] - 1;
            s_pages[b] = pages;
            s_partial[b] = rem;
        }
        my_tiles += splits[i] * Hkv;
        my_full += fulls[i] * Hkv;
    }
    int total_tiles, total_full;
    int start = block_exclusive_scan(my_tiles, &total_tiles, warp_sums);
    int full_start = block_exclusive_scan(my_full, &total_full, warp_sums);
    if (total_tiles > p.queue_cap) {
        if (tid == 0) {
            atomicOr(p.status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
            *p.tiles = 0;
        }
        return;
    }
    // ---- queue, row table and the full-tile part of the hand-out order
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        const int b = r0 + i;
        if (b >= B) continue;
        const int S = splits[i], F = fulls[i], pages = s_pages[b];
        p.row_start[b] = start;
        p.row_splits[b] = S;
        for (int kvh = 0; kvh < Hkv; ++kvh)
            for (int s = 0; s < S; ++s) {
                const int t = start + kvh * S + s;
                p.queue[t] = pkv_work_item{b, kvh, s, s * C, min((s + 1) * C, pages)};
                if (s < F) p.order[full_start + kvh * F + s] = t;
            }
        start += S * Hkv;
        full_start += F * Hkv;
    }
    __syncthreads();   // s_partial complete
    // ---- the partial tiles: rows ranked by their last tile's size (desc), then row
#pragma unroll
    for (int i = 0; i < kRowsPerThread; ++i) {
        const int b = r0 + i;
        if (b >= B || s_partial[b] == 0) continue;
        const int mine = s_partial[b];
        int before = 0;
        for (int c = 0; c < B; ++c) {
            const int other = s_partial[c];
            before += (other > mine) || (other == mine && other != 0 && c < b);
        }
        const int S = splits[i];
        const int row_start = p.row_start[b];
        for (int kvh = 0; kvh < Hkv; ++kvh)
            p.order[total_full + before * Hkv + kvh] = row_start + kvh * S + (S - 1);
    }
    if (tid == 0) *p.tiles = total_tiles;
}

}  // namespace devplan
}  // namespace pkv

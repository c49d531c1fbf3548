// pkv_devplan.cu -- the planner of a continuous-decoding step, on the device.
//
// The host planner (pkv_api.cpp) follows "PersistentKV: Page-Aware Decode
// Scheduling for Long-Context LLM Serving on Commodity GPUs" (gist.science
// summary), Methodology section 1 ("Row-Local Bounds", "Compact Workqueue"):
// tiles come from each row's true length and only non-empty
// (row, KV head, split) tiles are listed.  This kernel computes the same plan
// on the GPU, so that a whole step of continuous decoding (page allocation,
// plan, append, decode) runs without the host and can be captured once in a
// CUDA graph and replayed: the fixed-shape, fixed-address form that the "Fast
// Embeddings on GPUs" lesson (engineermaxxing, the CUDA-graph section) asks of
// a capturable step, with the dynamic decision moved into the kernel.
//
// One CTA of 1024 threads, for the lengths *before* the step's append:
//   1. page allocation: every row whose next token starts a page with no table
//      entry yet takes the next page of the device free list, in row order
//      (the host pool's FIFO rule, so tables come out identical);
//   2. the plan for the lengths after the append, with a fixed chunk of C
//      pages: S_b = ceil(P_b / C) splits, row_start = exclusive prefix sum of
//      S_b * Hkv, queue in lexicographic (b, kvh, s) order;
//   3. the persistent route's hand-out order: tiles by descending page count,
//      ties in queue order -- the host planner's stable sort, built here as
//      "all full-chunk tiles in queue order, then each row's last, partial
//      tile ranked by its size (ties by row, then KV head)".
// Rows are limited to kDevPlanMaxRows; sizes that do not fit the buffers set a
// status bit and leave the step's plan empty (the decode then writes NaN).
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 1024;
constexpr int kRowsPerThread = kDevPlanMaxRows / kThreads;

// Exclusive prefix sum over the CTA of one int per thread; returns the thread's
// prefix and writes the total to *total.
__device__ int block_exclusive_scan(int v, int* total) {
    __shared__ int warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
    *total = warp_sums[31];
    __syncthreads();
    return before;
}

__global__ void __launch_bounds__(kThreads) plan_step_kernel(const DevPlanParams p) {
    __shared__ int s_pages[kDevPlanMaxRows];   // P_b after the append
    __shared__ int s_partial[kDevPlanMaxRows]; // size of the row's last tile if partial, else 0
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
        if (b < B) {
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
    int rank = block_exclusive_scan(my_need, &total_need);
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
            const int n = max(p.lens[b], 0) + 1;
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
    int start = block_exclusive_scan(my_tiles, &total_tiles);
    int full_start = block_exclusive_scan(my_full, &total_full);
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

}  // namespace

cudaError_t launch_plan_step(const DevPlanParams& p, cudaStream_t stream) {
    plan_step_kernel<<<1, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv

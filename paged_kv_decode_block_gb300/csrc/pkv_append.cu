// pkv_append.cu -- write one new K/V token per row into its page.
//
// Layout from "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM
// Serving on Commodity GPUs" (gist.science summary), Methodology section 1
// "Layout": token t of row b lives in page block_table[b][t / page_size], slot
// t % page_size.  The operation is the KV-cache update of "GPUOS" (arXiv
// 2604.17861, section 4 operator library): the new token goes to position
// seq_lens[b], then the length grows by one.
//
// One CTA per row; each thread moves 16-byte vectors of the row's
// Hkv * D bf16 K and V values.  A row whose position has no page (table full,
// or the entry unassigned) sets PKV_DEV_ROW_FULL, one whose entry names a page
// outside the pool sets PKV_DEV_PAGE_OOB; either row is left unchanged.  The step variant
// (append_step_kernel) also enters the rows' new pages in the table and moves
// the step's plan from mapped pinned host memory into device memory, so that a
// host-planned session step needs no copy-engine transfer.  Rows marked idle in
// an `active` mask (slots of a session between an eviction and an admission)
// are skipped.  The slot kernels apply a batch of admissions and evictions
// (pkv_slots.cuh).
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv_internal.h"
#include "pkv_slots.cuh"

namespace pkv {
namespace {

constexpr int kSlotCopyCtas = 256;   // grid of the prompt copy (grid-stride over the tokens)

// Append the new token of row b (all threads of the CTA).  `new_idx` / `new_page`:
// a table entry to fill first (new_idx -1: none).
__device__ __forceinline__ void append_row(const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                                           uint16_t* __restrict__ k_pages, uint16_t* __restrict__ v_pages,
                                           int32_t* block_table, int32_t* __restrict__ seq_lens, int b, int Hkv,
                                           int D, int page_size, int max_pages, int num_pages, uint32_t* status,
                                           int new_idx, int new_page) {
    __shared__ int s_page, s_pos;
    if (threadIdx.x == 0) {
        const int pos = seq_lens[b];
        int page = -1;
        if (pos < 0 || pos / page_size >= max_pages) {
            atomicOr(status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));
        } else {
            int32_t* entry = block_table + static_cast<size_t>(b) * max_pages + pos / page_size;
            if (new_idx >= 0 && new_idx == pos / page_size) {
                *entry = new_page;
                page = new_page;
            } else {
                page = *entry;
            }
            if (page < 0) {   // no page assigned for the new position
                atomicOr(status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));
                page = -1;
            } else if (page >= num_pages) {
                atomicOr(status, static_cast<uint32_t>(PKV_DEV_PAGE_OOB));
                page = -1;
            }
        }
        s_page = page;
        s_pos = pos;
    }
    __syncthreads();
    if (s_page < 0) return;
    const int row = Hkv * D;   // elements of one token across all KV heads
    const size_t dst = (static_cast<size_t>(s_page) * page_size + s_pos % page_size) * row;
    const size_t src = static_cast<size_t>(b) * row;
    for (int c = threadIdx.x * 8; c < row; c += blockDim.x * 8) {
        *reinterpret_cast<uint4*>(k_pages + dst + c) = *reinterpret_cast<const uint4*>(k_new + src + c);
        *reinterpret_cast<uint4*>(v_pages + dst + c) = *reinterpret_cast<const uint4*>(v_new + src + c);
    }
    if (threadIdx.x == 0) seq_lens[b] = s_pos + 1;
}

__global__ void __launch_bounds__(128) append_kernel(const uint16_t* __restrict__ k_new,
                                                     const uint16_t* __restrict__ v_new,
                                                     uint16_t* __restrict__ k_pages, uint16_t* __restrict__ v_pages,
                                                     const int32_t* __restrict__ block_table,
                                                     int32_t* __restrict__ seq_lens, int Hkv, int D, int page_size,
                                                     int max_pages, int num_pages, uint32_t* status,
                                                     const int32_t* __restrict__ active) {
    if (active && !active[blockIdx.x]) return;   // an idle slot
    append_row(k_new, v_new, k_pages, v_pages, const_cast<int32_t*>(block_table), seq_lens, blockIdx.x, Hkv, D,
               page_size, max_pages, num_pages, status, -1, -1);
}

__global__ void __launch_bounds__(32) slot_apply_kernel(const SlotParams p) {
    if (threadIdx.x == 0) slots::apply_requests(p);
}

__global__ void __launch_bounds__(256) slot_copy_kernel(const SlotParams p) {
    slots::copy_prompts(p, static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                        static_cast<int64_t>(gridDim.x) * blockDim.x);
}

__global__ void __launch_bounds__(128) append_step_kernel(const AppendStepParams p) {
    // the step's plan: pinned host staging -> the plan's device buffer, 16 bytes
    // per thread where both ends allow it (both are 256-byte aligned allocations)
    if (p.plan_src) {
        const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        const int64_t nth = static_cast<int64_t>(gridDim.x) * blockDim.x;
        const int64_t n4 = p.plan_words / 4;
        const int4* src4 = reinterpret_cast<const int4*>(p.plan_src);
        int4* dst4 = reinterpret_cast<int4*>(p.plan_dst);
        for (int64_t i = tid; i < n4; i += nth) dst4[i] = src4[i];
        for (int64_t i = n4 * 4 + tid; i < p.plan_words; i += nth) p.plan_dst[i] = p.plan_src[i];
    }
    const int b = blockIdx.x;
    if (p.active && !p.active[b]) return;   // an idle slot
    const int new_idx = p.new_pages[2 * b], new_page = p.new_pages[2 * b + 1];
    append_row(p.k_new, p.v_new, p.k_pages, p.v_pages, p.block_table, p.seq_lens, b, p.Hkv, p.D, p.page_size,
               p.max_pages, p.num_pages, p.status, new_idx, new_page);
}

}  // namespace

cudaError_t launch_append(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_pages, uint16_t* v_pages,
                          const int32_t* block_table, int32_t* seq_lens, int B, int Hkv, int D, int page_size,
                          int max_pages, int num_pages, uint32_t* status, cudaStream_t stream,
                          const int32_t* active) {
    if (B == 0) return cudaSuccess;
    append_kernel<<<B, 128, 0, stream>>>(k_new, v_new, k_pages, v_pages, block_table, seq_lens, Hkv, D, page_size,
                                         max_pages, num_pages, status, active);
    return cudaGetLastError();
}

cudaError_t launch_slot_requests(const SlotParams& p, cudaStream_t stream) {
    if (p.n <= 0) return cudaSuccess;
    slot_apply_kernel<<<1, 32, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    slot_copy_kernel<<<kSlotCopyCtas, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_append_step(const AppendStepParams& p, cudaStream_t stream) {
    if (p.B == 0) return cudaSuccess;
    append_step_kernel<<<p.B, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv

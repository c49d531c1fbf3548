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
// One CTA of 1024 threads (the resident kernel runs the same code on one of
// its 256-thread CTAs), rows one per thread, for the lengths *before* the
// step's append:
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

#include "pkv_devplan.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kPlanThreads = 1024;

__global__ void __launch_bounds__(kPlanThreads) plan_step_kernel(const DevPlanParams p) {
    __shared__ int scratch[devplan::kPlanScratchInts];
    devplan::plan_step<kPlanThreads>(p, scratch);
}

}  // namespace

cudaError_t launch_plan_step(const DevPlanParams& p, cudaStream_t stream) {
    plan_step_kernel<<<1, kPlanThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv

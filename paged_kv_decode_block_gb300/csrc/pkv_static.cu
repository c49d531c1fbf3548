// pkv_static.cu -- paged decode attention without any device allocation.
//
// pkv_decode needs a plan, and pkv_plan allocates device memory (queue, split
// workspace, counters).  Some callers cannot allocate at call time: code that
// runs inside another framework's memory budget, real-time loops that must not
// touch the allocator, or hosts that forbid cudaMalloc after start-up.
// pkv_decode_static serves them: it runs the padded split route (one CTA per
// (row, KV head, split) slot of the B * Hkv * S_max grid, split ranges taken
// from the device lengths, merge fused into the last-arriving split) with its
// workspace in one file-scope __device__ array of kStaticScratchBytes.  The
// caller passes only inputs and outputs.
//
// Set-up: the array's host-side name is only a stand-in for the device
// object, so its device address is fetched with cudaGetSymbolAddress on the
// first call made while a device is current, and kept for that device's
// current context (keyed by the context's unique id, so a device reset, which
// brings a new context and reloads the module, triggers a fresh look-up).  That
// first call should therefore come before any stream capture.
//
// Sharing: every call on a device uses the same array, which keeps the last
// call's contents.  The counters that must start at zero are cleared on the
// stream at the start of each call.  Calls whose work overlaps on the GPU (two
// streams, or two host threads) race on the array and give wrong results; order
// them on one stream.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchAddr {
    unsigned long long ctx_id;   // unique id of the context the address belongs to (0: none yet)
    uint8_t* addr;
};
ScratchAddr g_scratch_addr[kMaxDevices] = {};

// Unique id of the calling thread's current context (cuCtxGetCurrent +
// cuCtxGetId, reached through the runtime's driver entry points); 0 if the
// driver does not provide them.
unsigned long long current_context_id() {
    typedef CUresult (*GetCurrentFn)(CUcontext*);
    typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Padded route row table: slots of row b start at b * Hkv * S_max, S_max each.
__global__ void fill_padded_rows(int32_t* row_start, int32_t* row_splits, int B, int Hkv, int s_max) {
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < B; b += gridDim.x * blockDim.x) {
        row_start[b] = b * Hkv * s_max;
        row_splits[b] = s_max;
    }
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace
}  // namespace pkv

extern "C" int pkv_decode_static(const void* q, const void* k_pages, const void* v_pages,
                                 const int32_t* block_table_d, const int32_t* seq_lens_d, int32_t page_size,
                                 const pkv_geom* g, int32_t max_seq_len, int32_t num_splits, float* out, float* lse,
                                 pkv_stream_t stream) {
    using namespace pkv;
    if (!g || g->batch < 0 || g->num_q_heads <= 0 || g->num_kv_heads <= 0 || g->max_pages_per_seq <= 0 ||
        g->num_pages <= 0 || page_size <= 0 || max_seq_len < 0 || num_splits <= 0 ||
        g->num_q_heads % g->num_kv_heads != 0)
        return PKV_EINVAL;
    if (page_size % kBlockRows != 0 || page_size > 256) return PKV_EUNSUPPORTED;
    const int G = g->num_q_heads / g->num_kv_heads;
    if (!shape_supported(g->head_dim, G)) return PKV_EUNSUPPORTED;
    if (static_cast<int64_t>(g->num_pages) * page_size > INT32_MAX ||
        static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(g->max_pages_per_seq) * page_size)
        return PKV_EINVAL;
    if (g->batch == 0) return PKV_OK;
    if (!q || !k_pages || !v_pages || !block_table_d || !seq_lens_d || !out || !lse) return PKV_EINVAL;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_pages) |
                          reinterpret_cast<uintptr_t>(v_pages) | reinterpret_cast<uintptr_t>(out);
    if ((mis & 15u) || (reinterpret_cast<uintptr_t>(lse) & 3u)) return PKV_EINVAL;

    // split geometry from the length bound: chunk C pages, S_max slots per (row, KV head)
    const int64_t p_max = ceil_div(max_seq_len, page_size);
    int64_t chunk = p_max > 0 ? ceil_div(p_max, num_splits) : 1;
    chunk = std::max<int64_t>(chunk, ceil_div(p_max, kMergeCapFloats / G));
    const int64_t s_max = std::max<int64_t>(1, ceil_div(p_max, chunk));
    const int64_t B = g->batch, Hkv = g->num_kv_heads, D = g->head_dim;
    const int64_t slots = B * Hkv * s_max;

    // layout of the scratch array
    const size_t off_arrive = 256;   // DeviceCounters live at offset 0
    const size_t off_rows = off_arrive + round256(B * Hkv * sizeof(uint32_t));
    const size_t off_lse = off_rows + round256(2 * B * sizeof(int32_t));
    const size_t off_o = off_lse + round256(slots * G * sizeof(float));
    const size_t total = off_o + static_cast<size_t>(slots) * G * D * sizeof(float);
    if (total > kStaticScratchBytes) return PKV_ENOSPACE;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
    uint8_t* base = nullptr;
    {
        // the first call with this device current (in this context) looks the
        // array's device address up; a context without an id is looked up every call
        const unsigned long long ctx_id = current_context_id();
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        ScratchAddr& slot = g_scratch_addr[dev];
        if (ctx_id == 0 || slot.ctx_id != ctx_id || !slot.addr) {
            void* addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_static_scratch);
            if (e != cudaSuccess) return cuda_fail(e);
            if (!addr) return cuda_fail(cudaErrorInvalidSymbol);
            slot.addr = static_cast<uint8_t*>(addr);
            slot.ctx_id = ctx_id;
        }
        base = slot.addr;
    }

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    AttnParams a{};
    a.q = static_cast<const uint16_t*>(q);
    a.k_pages = static_cast<const uint16_t*>(k_pages);
    a.v_pages = static_cast<const uint16_t*>(v_pages);
    a.block_table = block_table_d;
    a.seq_lens = seq_lens_d;
    a.queue = nullptr;
    a.row_start = reinterpret_cast<const int32_t*>(base + off_rows);
    a.row_splits = a.row_start + B;
    a.out = out;
    a.lse = lse;
    a.ws_o = reinterpret_cast<float*>(base + off_o);
    a.ws_lse = reinterpret_cast<float*>(base + off_lse);
    a.arrive = reinterpret_cast<uint32_t*>(base + off_arrive);
    a.ctr = reinterpret_cast<DeviceCounters*>(base);
    a.B = g->batch;
    a.Hq = g->num_q_heads;
    a.Hkv = g->num_kv_heads;
    a.D = g->head_dim;
    a.page_size = page_size;
    a.max_pages = g->max_pages_per_seq;
    a.num_pages = g->num_pages;
    a.chunk_pages = static_cast<int32_t>(chunk);
    a.max_splits = static_cast<int32_t>(s_max);
    a.num_tiles = static_cast<int32_t>(slots);
    a.route = kRoutePadded;
    a.fused_merge = 1;
    a.use_mma = 1;
    a.copy_lsu = 1;   // cp.async staging: the TMA descriptors below are never read
    a.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(D)));

    // arrival counters and the status word must start at zero
    e = cudaMemsetAsync(base, 0, off_rows, s);
    if (e != cudaSuccess) return cuda_fail(e);
    // the launch's own result (an earlier, unrelated error is not picked up here)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    e = cudaLaunchKernelEx(&cfg, fill_padded_rows, const_cast<int32_t*>(a.row_start),
                           const_cast<int32_t*>(a.row_splits), static_cast<int>(g->batch),
                           static_cast<int>(g->num_kv_heads), static_cast<int>(s_max));
    if (e != cudaSuccess) return cuda_fail(e);
    CUtensorMap unused;
    memset(&unused, 0, sizeof(unused));
    e = launch_attention(a, unused, unused, static_cast<int>(slots), s);
    if (e != cudaSuccess) return cuda_fail(e);
    return PKV_OK;
}

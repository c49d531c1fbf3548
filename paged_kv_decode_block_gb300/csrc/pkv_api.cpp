// pkv_api.cpp -- host side of pkv: validation, the adaptive policy, the work
// planner, plan memory, kernel launches and the page pool, behind the C ABI
// declared in include/pkv.h.
//
// Planner and policy follow "PersistentKV: Page-Aware Decode Scheduling for
// Long-Context LLM Serving on Commodity GPUs" (gist.science summary),
// Technical Summary:
//   * Methodology section 1 "Row-Local Bounds" / "Compact Workqueue": split
//     ranges come from each row's true length; the queue lists only non-empty
//     (row, KV head, split) tiles;
//   * Methodology section 2 "Calibrated Adaptive Policy": the route is chosen
//     from the batch and the longest context.  Its thresholds were fitted to a
//     28-SM GPU; here they are restated in SM units: a batch whose B * Hkv
//     (row, KV head) units already fill `direct_units_per_sm` CTAs per SM runs
//     the single-pass DIRECT kernel (the summary's high-batch route), anything
//     smaller is split into the smallest page chunks whose tiles still fit one
//     wave of `target_ctas_per_sm` CTAs per SM.
// Split rule (the summary states none exactly): boundaries on pages, one chunk
// of C pages per plan, row b gets S_b = ceil(P_b / C) splits, split s covers
// pages [s*C, min((s+1)*C, P_b)); a requested split count S gives
// C = ceil(P_max / S).  Queue order is lexicographic in (b, kvh, s).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <deque>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "pkv.h"
#include "pkv_internal.h"

static_assert(PKV_TRACE_WORDS == pkv::kTraceWords, "trace row layout");

namespace {
thread_local int g_last_cuda_error = 0;
}  // namespace

namespace pkv {
int cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return PKV_ECUDA;
}
}  // namespace pkv
using pkv::cuda_fail;

namespace {

// An NVTX range over one library call, so that a profiler's timeline shows the
// host side of each call (planning, staging, launches).  Without a profiler
// attached a push or pop is one test of a null function pointer.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};


#define PKV_CUDA(call)                                 \
    do {                                               \
        cudaError_t e_ = (call);                       \
        if (e_ != cudaSuccess) return cuda_fail(e_);   \
    } while (0)

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Options {
    int force_mode = PKV_MODE_AUTO;
    int num_splits = 0;
    int direct_units_per_sm = 2;
    int target_ctas_per_sm = 2;
    int min_chunk_pages = 8;
    int ctas_per_sm = 0;
    int separate_merge = 0;
    int num_sms = 0;
    int math = PKV_MATH_AUTO;
    int copy = PKV_COPY_AUTO;
    int merge = PKV_MERGE_AUTO;
};

int resolve_options(const pkv_plan_opts* o, Options* r) {
    if (!o) return PKV_OK;
    if (o->force_mode < PKV_MODE_AUTO || o->force_mode > PKV_MODE_PERSISTENT) return PKV_EINVAL;
    if (o->num_splits < 0 || o->direct_units_per_sm < 0 || o->target_ctas_per_sm < 0 ||
        o->min_chunk_pages < 0 || o->ctas_per_sm < 0 || o->num_sms < 0 || o->separate_merge < 0 ||
        o->separate_merge > 1 || o->math < PKV_MATH_AUTO || o->math > PKV_MATH_MMA || o->copy < PKV_COPY_AUTO ||
        o->copy > PKV_COPY_TMA || o->merge < PKV_MERGE_AUTO || o->merge > PKV_MERGE_ALL)
        return PKV_EINVAL;
    r->merge = o->merge;
    r->math = o->math;
    r->copy = o->copy;
    r->force_mode = o->force_mode;
    r->num_splits = o->num_splits;
    if (o->direct_units_per_sm) r->direct_units_per_sm = o->direct_units_per_sm;
    if (o->target_ctas_per_sm) r->target_ctas_per_sm = o->target_ctas_per_sm;
    if (o->min_chunk_pages) r->min_chunk_pages = o->min_chunk_pages;
    r->ctas_per_sm = o->ctas_per_sm;
    r->separate_merge = o->separate_merge;
    r->num_sms = o->num_sms;
    return PKV_OK;
}

int validate_geometry(const pkv_geom* g, int32_t page_size) {
    if (!g) return PKV_EINVAL;
    if (g->batch < 0 || g->num_q_heads <= 0 || g->num_kv_heads <= 0 || g->head_dim <= 0 ||
        g->max_pages_per_seq <= 0 || g->num_pages <= 0 || page_size <= 0)
        return PKV_EINVAL;
    if (g->num_q_heads % g->num_kv_heads != 0) return PKV_EINVAL;
    if (static_cast<int64_t>(g->num_pages) * page_size > INT32_MAX) return PKV_EINVAL;
    if (static_cast<int64_t>(g->max_pages_per_seq) * page_size > INT32_MAX) return PKV_EINVAL;
    if (page_size % pkv::kBlockRows != 0 || page_size > 256) return PKV_EUNSUPPORTED;
    if (!pkv::shape_supported(g->head_dim, g->num_q_heads / g->num_kv_heads)) return PKV_EUNSUPPORTED;
    return PKV_OK;
}

int validate_rows(const pkv_geom& g, int32_t page_size, const int32_t* lens, const int32_t* table) {
    if (g.batch > 0 && !lens) return PKV_EINVAL;
    const int64_t cap = static_cast<int64_t>(g.max_pages_per_seq) * page_size;
    for (int b = 0; b < g.batch; ++b) {
        if (lens[b] < 0 || lens[b] > cap) return PKV_EINVAL;
        if (table) {
            const int64_t pages = ceil_div(lens[b], page_size);
            const int32_t* row = table + static_cast<size_t>(b) * g.max_pages_per_seq;
            for (int64_t i = 0; i < pages; ++i)
                if (row[i] < 0 || row[i] >= g.num_pages) return PKV_EINVAL;
        }
    }
    return PKV_OK;
}

// Everything the planner decides, computed on the host only.
struct Plan {
    int32_t mode = PKV_MODE_DIRECT;
    int32_t chunk = 1;
    int32_t s_max = 0;
    int32_t grid = 0;
    int32_t empty_tiles = 0;
    bool need_merge = false;
    bool any_empty_row = false;   // some row has no tokens
    int32_t merge = 0;   // pkv_plan_info.merge
    int32_t ws_slots = 0;
    int64_t kv_bytes = 0, ws_bytes = 0, table_bytes = 0;
    std::vector<pkv_work_item> items;   // queue (or padded grid / direct tiles, for inspection)
    std::vector<int32_t> row_start, row_splits;
    std::vector<int32_t> order;         // persistent route: queue indices, longest tile first
};

// `resident_ctas`: attention CTAs the device holds at once (a cooperative
// launch of up to this many is possible).
int compute_plan(const pkv_geom& g, int32_t ps, const int32_t* lens, const Options& o, int num_sms,
                 int ctas_per_sm, int64_t resident_ctas, Plan* r) {
    const int B = g.batch, Hkv = g.num_kv_heads, G = g.num_q_heads / g.num_kv_heads, D = g.head_dim;
    std::vector<int32_t> pages(B);
    int64_t p_max = 0, p_total = 0, tokens = 0;
    for (int b = 0; b < B; ++b) {
        pages[b] = static_cast<int32_t>(ceil_div(lens[b], ps));
        p_max = std::max<int64_t>(p_max, pages[b]);
        p_total += pages[b];
        tokens += lens[b];
    }
    const int64_t units = static_cast<int64_t>(B) * Hkv;
    const bool big_batch = units >= static_cast<int64_t>(o.direct_units_per_sm) * num_sms;
    // Smallest chunk (most parallelism) whose tiles still fit one wave of
    // target_ctas_per_sm CTAs per SM: ceil() per row adds up to one tile per
    // (row, KV head) beyond Hkv * P_total / C, and a second, mostly empty wave
    // would cost as much as the first.
    auto policy_chunk = [&]() -> int64_t {
        if (big_batch) return std::max<int64_t>(p_max, 1);
        const int64_t target = std::max<int64_t>(1, static_cast<int64_t>(o.target_ctas_per_sm) * num_sms);
        int64_t c = std::max<int64_t>(o.min_chunk_pages, ceil_div(Hkv * p_total, target));
        while (c < p_max) {
            int64_t tiles = 0;
            for (int b = 0; b < B; ++b) tiles += Hkv * ceil_div(pages[b], c);
            if (tiles <= target) break;
            ++c;
        }
        return c;
    };

    int64_t chunk;
    int mode = o.force_mode;
    if (o.num_splits > 0)
        chunk = p_max > 0 ? ceil_div(p_max, o.num_splits) : 1;
    else if (mode == PKV_MODE_DIRECT)
        chunk = std::max<int64_t>(p_max, 1);
    else
        chunk = policy_chunk();
    chunk = std::max<int64_t>(chunk, 1);
    // an exact merge holds all splits of one (row, KV head) in shared memory
    chunk = std::max<int64_t>(chunk, ceil_div(p_max, pkv::kMergeCapFloats / G));
    // A small batch whose rows fit one chunk still takes the queue route (one
    // split per row, finalised in place): its host-staged tiles start before the
    // grid dependency wait.  On rows of up to 8 pages it measured as fast as
    // DIRECT or one timer step (about 2 us) faster, never slower.
    if (mode == PKV_MODE_AUTO) mode = chunk >= p_max && big_batch ? PKV_MODE_DIRECT : PKV_MODE_SPLIT_QUEUE;
    if (mode == PKV_MODE_DIRECT) chunk = std::max<int64_t>(p_max, 1);

    r->mode = mode;
    r->chunk = static_cast<int32_t>(chunk);
    r->s_max = static_cast<int32_t>(ceil_div(p_max, chunk));
    r->kv_bytes = tokens * Hkv * D * 2 * 2;
    r->table_bytes = p_total * Hkv * 4;
    r->items.clear();
    r->order.clear();   // only the compact-queue routes hand tiles out in an order
    r->row_start.assign(B, 0);
    r->row_splits.assign(B, 0);
    r->empty_tiles = 0;
    r->need_merge = false;
    r->any_empty_row = std::any_of(pages.begin(), pages.end(), [](int32_t n) { return n == 0; });
    int64_t merged_slots = 0;

    if (mode == PKV_MODE_DIRECT) {
        for (int b = 0; b < B; ++b)
            for (int kvh = 0; kvh < Hkv; ++kvh) r->items.push_back({b, kvh, 0, 0, pages[b]});
        r->grid = B * Hkv;
        r->ws_slots = 0;
    } else if (mode == PKV_MODE_SPLIT_PADDED) {
        r->s_max = std::max(r->s_max, 1);   // an all-empty batch still gets one (neutral) slot per row
        for (int b = 0; b < B; ++b) {
            r->row_start[b] = b * Hkv * r->s_max;
            r->row_splits[b] = r->s_max;
            for (int kvh = 0; kvh < Hkv; ++kvh)
                for (int s = 0; s < r->s_max; ++s) {
                    const int32_t pb = static_cast<int32_t>(std::min<int64_t>(s * chunk, pages[b]));
                    const int32_t pe = static_cast<int32_t>(std::min<int64_t>((s + 1) * chunk, pages[b]));
                    if (pb == pe) ++r->empty_tiles;
                    r->items.push_back({b, kvh, s, pb, pe});
                }
        }
        r->grid = B * Hkv * r->s_max;
        r->ws_slots = r->grid;
        r->need_merge = o.separate_merge && r->s_max != 1;
        if (r->s_max != 1) merged_slots = r->grid;
    } else {   // compact queue: SPLIT_QUEUE and PERSISTENT
        int32_t slot = 0;
        bool any_unfinished = false;
        for (int b = 0; b < B; ++b) {
            const int32_t sb = static_cast<int32_t>(ceil_div(pages[b], chunk));
            r->row_start[b] = slot;
            r->row_splits[b] = sb;
            if (sb != 1) any_unfinished = true;
            if (sb > 1) merged_slots += static_cast<int64_t>(sb) * Hkv;
            for (int kvh = 0; kvh < Hkv; ++kvh)
                for (int s = 0; s < sb; ++s)
                    r->items.push_back({b, kvh, s, static_cast<int32_t>(s * chunk),
                                        static_cast<int32_t>(std::min<int64_t>((s + 1) * chunk, pages[b]))});
            slot += sb * Hkv;
        }
        r->ws_slots = slot;
        const int32_t T = static_cast<int32_t>(r->items.size());
        // rows with no tokens have no tiles; the attention kernel writes their
        // neutral state (a fused merge) or the merge kernel does (separate)
        if (mode == PKV_MODE_SPLIT_QUEUE)
            r->grid = B > 0 ? std::max<int32_t>(T, 1) : 0;
        else
            r->grid = B > 0 ? std::max(1, std::min<int32_t>(T, num_sms * std::max(1, ctas_per_sm))) : 0;
        r->need_merge = o.separate_merge && any_unfinished;
        // The persistent grid hands tiles out in this order: longest first (ties in
        // queue order), so that the long tiles do not start last and set the tail.
        r->order.resize(T);
        for (int32_t t = 0; t < T; ++t) r->order[t] = t;
        if (mode == PKV_MODE_PERSISTENT)
            std::stable_sort(r->order.begin(), r->order.end(), [&](int32_t a, int32_t b) {
                return r->items[a].page_end - r->items[a].page_begin > r->items[b].page_end - r->items[b].page_begin;
            });
    }
    r->ws_bytes = merged_slots * G * (D + 1) * 4 * 2;   // written once, read once
    // How the merge of the split partials is shared out
    r->merge = 0;
    if (merged_slots > 0) {
        if (o.separate_merge) {
            r->merge = 3;
        } else {
            const bool one_wave = (mode == PKV_MODE_SPLIT_QUEUE || mode == PKV_MODE_SPLIT_PADDED) &&
                                  static_cast<int64_t>(r->grid) <= resident_ctas;
            // AUTO takes LAST: its launch overlaps the previous kernel's tail
            // (programmatic dependent launch), which a cooperative launch does
            // not; back to back that is worth more than ALL's shorter merge.
            if (o.merge == PKV_MERGE_ALL && !one_wave) return PKV_EUNSUPPORTED;
            r->merge = o.merge == PKV_MERGE_ALL ? PKV_MERGE_ALL : PKV_MERGE_LAST;
        }
    }
    return PKV_OK;
}

int32_t launches_of(const Plan& p) { return (p.grid > 0 ? 1 : 0) + (p.need_merge ? 1 : 0); }

// How K/V reach shared memory for a plan: AUTO takes TMA boxes on the
// one-tile-per-CTA routes and cp.async on the persistent route (each measured
// faster there).
int32_t resolved_copy(const Options& o, int32_t mode) {
    if (o.copy != PKV_COPY_AUTO) return o.copy;
    return mode == PKV_MODE_PERSISTENT ? PKV_COPY_LSU : PKV_COPY_TMA;
}

void fill_info(const Plan& p, const pkv_geom& g, int num_sms, const Options& o, pkv_plan_info* info) {
    memset(info, 0, sizeof(*info));
    info->mode = p.mode;
    info->chunk_pages = p.chunk;
    info->max_splits = p.s_max;
    info->num_tiles = p.grid;
    if (p.mode == PKV_MODE_PERSISTENT) info->num_tiles = static_cast<int32_t>(p.items.size());
    info->num_work_items = static_cast<int32_t>(p.items.size());
    info->empty_tiles = p.empty_tiles;
    info->launches_per_step = g.batch > 0 ? launches_of(p) : 0;
    info->grid_ctas = p.grid;
    info->num_sms = num_sms;
    info->merge = p.merge;
    info->kv_bytes = p.kv_bytes;
    info->workspace_bytes = p.ws_bytes;
    info->table_bytes = p.table_bytes;
    info->copy = resolved_copy(o, p.mode);
}

// ------------------------------------------------------------------ TMA descriptors

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// The pool [num_pages][page_size][Hkv][D] bf16 as a 3-D tensor
// {D, Hkv, num_pages * page_size} (innermost first); one box is 64 elements
// (128 B) of kBlockRows consecutive tokens of one KV head, stored with the
// 128-byte swizzle the kernels' shared-memory addressing expects.
int encode_pool_map(CUtensorMap* map, const void* pool, const pkv_geom& g, int32_t page_size) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cuda_fail(cudaErrorNotSupported);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(g.head_dim), static_cast<cuuint64_t>(g.num_kv_heads),
                                static_cast<cuuint64_t>(g.num_pages) * page_size};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.head_dim) * 2,
                                   static_cast<cuuint64_t>(g.num_kv_heads) * g.head_dim * 2};
    const cuuint32_t box[3] = {64u, 1u, static_cast<cuuint32_t>(pkv::kBlockRows)};   // 128 B x 16 tokens
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The address through which the current device reaches host memory `h`, if
// `h` lies in pinned (page-locked, cudaMallocHost / cudaHostAlloc /
// cudaHostRegister) memory mapped for this device and that address has the
// given alignment; nullptr for pageable or unmapped memory.
const void* mapped_host_address(const void* h, uintptr_t align) {
    cudaPointerAttributes attr{};
    if (cudaPointerGetAttributes(&attr, h) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    if (attr.type != cudaMemoryTypeHost || !attr.devicePointer) return nullptr;
    if (reinterpret_cast<uintptr_t>(attr.devicePointer) & (align - 1)) return nullptr;
    return attr.devicePointer;
}

}  // namespace

// ------------------------------------------------------------------ plan object

struct pkv_plan_s {
    pkv_geom g{};
    int32_t page_size = 0;
    Options opts;
    int device = 0;
    int num_sms = 0;
    int ctas_per_sm = 1;
    int64_t resident_ctas = 0;   // attention CTAs the device holds at once
    Plan plan;
    Plan next;   // pkv_plan_update builds here, then swaps: a failed update leaves `plan` as it was

    // host staging (pinned) and device copy: [items][row_start B][row_splits B]
    int32_t* host_buf = nullptr;
    int32_t* dev_buf = nullptr;
    size_t buf_cap_items = 0;
    size_t upload_bytes = 0;
    bool dirty = false;
    cudaEvent_t upload_done = nullptr;
    bool upload_recorded = false;

    float* ws_o = nullptr;
    float* ws_lse = nullptr;
    size_t ws_cap_slots = 0;
    uint32_t* arrive = nullptr;
    pkv::DeviceCounters* ctr = nullptr;

    const void* map_k = nullptr;
    const void* map_v = nullptr;
    CUtensorMap kmap{}, vmap{};

    bool profile = false;
    cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
    int ev_launches = 0;

    // per-CTA timeline of the attention launch (pkv_trace_enable)
    bool trace_on = false;
    uint64_t* trace = nullptr;   // device [trace_cap][kTraceWords]
    int trace_cap = 0;           // rows allocated
    int trace_rows = 0;          // CTAs of the last traced launch

    // Device address of host_buf (pinned memory is mapped into the GPU's
    // address space), so pkv_decode_host can read a fresh plan in place.
    const int32_t* host_buf_dev = nullptr;

    // pkv_decode_host: pinned, device-mapped staging [q][out][lse] for host
    // buffers the GPU cannot address itself (allocated on first need)
    uint8_t* host_stage = nullptr;
    uint8_t* host_stage_dev = nullptr;
};

namespace {

void release(pkv_plan_s* p) {
    if (!p) return;
    if (p->upload_recorded) cudaEventSynchronize(p->upload_done);
    cudaFreeHost(p->host_buf);
    cudaFree(p->dev_buf);
    cudaFree(p->ws_o);
    cudaFree(p->ws_lse);
    cudaFree(p->arrive);
    cudaFree(p->ctr);
    cudaFree(p->trace);
    cudaFreeHost(p->host_stage);
    if (p->upload_done) cudaEventDestroy(p->upload_done);
    for (auto& e : p->ev)
        if (e) cudaEventDestroy(e);
    delete p;
}

// Size buffers for the current plan (grow only) and stage the queue for upload.
int stage(pkv_plan_s* p) {
    const Plan& pl = p->plan;
    const size_t items = pl.items.size();
    const int B = p->g.batch;
    if (items > p->buf_cap_items || !p->host_buf) {
        const size_t cap = std::max<size_t>(items + items / 2, 64);
        if (p->upload_recorded) PKV_CUDA(cudaEventSynchronize(p->upload_done));
        cudaFreeHost(p->host_buf);
        cudaFree(p->dev_buf);
        p->host_buf = nullptr;
        p->host_buf_dev = nullptr;
        p->dev_buf = nullptr;
        p->buf_cap_items = 0;
        const size_t bytes = (cap * 6 + 2 * static_cast<size_t>(B)) * sizeof(int32_t);
        if (cudaMallocHost(&p->host_buf, bytes) != cudaSuccess) return PKV_ENOMEM;
        if (cudaMalloc(&p->dev_buf, bytes) != cudaSuccess) return PKV_ENOMEM;
        void* mapped = nullptr;
        if (cudaHostGetDevicePointer(&mapped, p->host_buf, 0) == cudaSuccess)
            p->host_buf_dev = static_cast<const int32_t*>(mapped);
        else
            (void)cudaGetLastError();   // not mapped: pkv_decode_host uploads the plan instead
        p->buf_cap_items = cap;
    }
    const size_t slots = static_cast<size_t>(std::max(pl.ws_slots, 1));
    const int G = p->g.num_q_heads / p->g.num_kv_heads;
    if (slots > p->ws_cap_slots) {
        const size_t cap = slots + slots / 2;
        cudaFree(p->ws_o);
        cudaFree(p->ws_lse);
        p->ws_o = nullptr;
        p->ws_lse = nullptr;
        p->ws_cap_slots = 0;
        if (cudaMalloc(&p->ws_o, cap * G * p->g.head_dim * sizeof(float)) != cudaSuccess) return PKV_ENOMEM;
        if (cudaMalloc(&p->ws_lse, cap * G * sizeof(float)) != cudaSuccess) return PKV_ENOMEM;
        p->ws_cap_slots = cap;
    }
    // host staging: the queue, then row_start, row_splits, then the hand-out order
    int32_t* h = p->host_buf;
    memcpy(h, pl.items.data(), items * sizeof(pkv_work_item));
    int32_t* rs = h + p->buf_cap_items * 5;
    if (B > 0) {
        memcpy(rs, pl.row_start.data(), B * sizeof(int32_t));
        memcpy(rs + B, pl.row_splits.data(), B * sizeof(int32_t));
    }
    if (!pl.order.empty()) memcpy(rs + 2 * B, pl.order.data(), pl.order.size() * sizeof(int32_t));
    p->upload_bytes = (p->buf_cap_items * 6 + 2 * static_cast<size_t>(B)) * sizeof(int32_t);
    p->dirty = pl.mode != PKV_MODE_DIRECT;
    return PKV_OK;
}

}  // namespace

extern "C" {

const char* pkv_strerror(int code) {
    switch (code) {
        case PKV_OK: return "ok";
        case PKV_EINVAL: return "invalid argument";
        case PKV_ENOMEM: return "out of memory";
        case PKV_ECUDA: return "CUDA runtime error";
        case PKV_EUNSUPPORTED: return "unsupported shape";
        case PKV_EDEVICE: return "device status word set";
        case PKV_ENOSPACE: return "no free page / row table full";
        default: return "unknown error";
    }
}

int pkv_last_cuda_error(void) { return g_last_cuda_error; }

int pkv_plan_dry_run(const int32_t* seq_lens_h, const int32_t* block_table_h, int32_t page_size,
                     const pkv_geom* geom, const pkv_plan_opts* opts, pkv_plan_info* info,
                     pkv_work_item* items, int32_t capacity, int32_t* count) {
    NvtxRange range("pkv_plan_dry_run");
    Options o;
    int rc = resolve_options(opts, &o);
    if (rc) return rc;
    if ((rc = validate_geometry(geom, page_size))) return rc;
    if ((rc = validate_rows(*geom, page_size, seq_lens_h, block_table_h))) return rc;
    if (o.num_sms <= 0) return PKV_EINVAL;   // no device is consulted here
    Plan pl;
    if ((rc = compute_plan(*geom, page_size, seq_lens_h, o, o.num_sms, std::max(1, o.ctas_per_sm),
                           static_cast<int64_t>(o.num_sms) * std::max(1, o.ctas_per_sm), &pl)))
        return rc;
    if (info) fill_info(pl, *geom, o.num_sms, o, info);
    const int32_t n = static_cast<int32_t>(pl.items.size());
    if (count) *count = n;
    if (items && capacity > 0) memcpy(items, pl.items.data(), sizeof(pkv_work_item) * std::min(n, capacity));
    return PKV_OK;
}

int pkv_plan(const int32_t* seq_lens_h, const int32_t* block_table_h, int32_t page_size, const pkv_geom* geom,
             const pkv_plan_opts* opts, pkv_plan_t* plan) {
    NvtxRange range("pkv_plan");
    if (!plan) return PKV_EINVAL;
    *plan = nullptr;
    Options o;
    int rc = resolve_options(opts, &o);
    if (rc) return rc;
    if ((rc = validate_geometry(geom, page_size))) return rc;
    if ((rc = validate_rows(*geom, page_size, seq_lens_h, block_table_h))) return rc;

    pkv_plan_s* p = new (std::nothrow) pkv_plan_s;
    if (!p) return PKV_ENOMEM;
    p->g = *geom;
    p->page_size = page_size;
    p->opts = o;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e == cudaSuccess && o.num_sms <= 0)
        e = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, p->device);
    if (e != cudaSuccess) {
        delete p;
        return cuda_fail(e);
    }
    const int G = geom->num_q_heads / geom->num_kv_heads;
    {
        int dev_sms = 0;
        if (cudaDeviceGetAttribute(&dev_sms, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
            delete p;
            return cuda_fail(cudaGetLastError());
        }
        const int occ = pkv::attention_ctas_per_sm(geom->head_dim, G, o.math != PKV_MATH_FMA);
        p->resident_ctas = static_cast<int64_t>(dev_sms) * occ;
    }
    if (o.num_sms > 0) p->num_sms = o.num_sms;
    p->ctas_per_sm = o.ctas_per_sm > 0 ? o.ctas_per_sm
                                       : std::max(1, pkv::attention_ctas_per_sm(geom->head_dim, G,
                                                                                o.math != PKV_MATH_FMA));

    if ((rc = compute_plan(p->g, page_size, seq_lens_h, o, p->num_sms, p->ctas_per_sm, p->resident_ctas,
                           &p->plan))) {
        delete p;
        return rc;
    }
    if (cudaEventCreateWithFlags(&p->upload_done, cudaEventDisableTiming) != cudaSuccess ||
        cudaMalloc(&p->ctr, sizeof(pkv::DeviceCounters)) != cudaSuccess ||
        cudaMalloc(&p->arrive, 2 * sizeof(uint32_t) * std::max(1, geom->batch * geom->num_kv_heads)) != cudaSuccess) {
        release(p);
        return PKV_ENOMEM;
    }
    if (cudaMemset(p->ctr, 0, sizeof(pkv::DeviceCounters)) != cudaSuccess ||
        cudaMemset(p->arrive, 0, 2 * sizeof(uint32_t) * std::max(1, geom->batch * geom->num_kv_heads)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        release(p);
        return cuda_fail(cudaGetLastError());
    }
    if ((rc = stage(p))) {
        release(p);
        return rc;
    }
    *plan = p;
    return PKV_OK;
}

int pkv_plan_update(pkv_plan_t p, const int32_t* seq_lens_h, const int32_t* block_table_h) {
    NvtxRange range("pkv_plan_update");
    if (!p) return PKV_EINVAL;
    int rc = validate_rows(p->g, p->page_size, seq_lens_h, block_table_h);
    if (rc) return rc;
    if (p->upload_recorded) PKV_CUDA(cudaEventSynchronize(p->upload_done));
    if ((rc = compute_plan(p->g, p->page_size, seq_lens_h, p->opts, p->num_sms, p->ctas_per_sm, p->resident_ctas,
                           &p->next)))
        return rc;
    std::swap(p->plan, p->next);
    return stage(p);
}

void pkv_plan_destroy(pkv_plan_t p) { release(p); }

int pkv_plan_get_info(pkv_plan_t p, pkv_plan_info* info) {
    if (!p || !info) return PKV_EINVAL;
    fill_info(p->plan, p->g, p->num_sms, p->opts, info);
    return PKV_OK;
}

int pkv_plan_queue(pkv_plan_t p, pkv_work_item* items, int32_t capacity, int32_t* count) {
    if (!p || !count) return PKV_EINVAL;
    const int32_t n = static_cast<int32_t>(p->plan.items.size());
    *count = n;
    if (items && capacity > 0) memcpy(items, p->plan.items.data(), sizeof(pkv_work_item) * std::min(n, capacity));
    return PKV_OK;
}

}  // extern "C"

namespace {

// A plan built on the device for one step (see pkv_devplan.cu) instead of by
// the host planner: queue, row table, hand-out order and tile count all live
// in device memory, written by the planner kernel earlier on the stream.
struct DevicePlan {
    const pkv_work_item* queue;
    const int32_t* row_start;
    const int32_t* row_splits;
    const int32_t* order;
    const int32_t* tiles;
    int32_t chunk;
    int32_t max_splits;
};

// Everything a decode launch needs, checked: the pending plan upload is
// enqueued on `s`, the TMA maps follow the pools, and `a` / `grid` /
// `need_merge` describe the launch (over the device-built plan `dp` if given).
// How the host plan reaches the kernel (when it is not device-built).
enum class PlanSource {
    kUpload,        // copied to the device buffer on the stream if it changed (default)
    kInPlace,       // a plan not yet uploaded is read by the kernel from its pinned, mapped host
                    // staging (no copy; the upload stays pending for later launches): the caller
                    // must not change the plan before the launch has finished
    kKernelCopied   // an earlier kernel on the stream has copied it into the device buffer, so the
                    // attention kernel must not read it before its grid dependency wait
};

int prepare_decode(pkv_plan_t p, const void* q, const void* k_pages, const void* v_pages,
                   const int32_t* block_table_d, const int32_t* seq_lens_d, float* out, float* lse, cudaStream_t s,
                   const DevicePlan* dp, pkv::AttnParams* a_out, int* grid_out, bool* need_merge_out,
                   PlanSource src = PlanSource::kUpload) {
    if (!q || !k_pages || !v_pages || !block_table_d || !seq_lens_d || !out || !lse) return PKV_EINVAL;
    if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(block_table_d) & 3u) ||
        (reinterpret_cast<uintptr_t>(seq_lens_d) & 3u))
        return PKV_EINVAL;
    int dev = -1;
    PKV_CUDA(cudaGetDevice(&dev));
    if (dev != p->device) return PKV_EINVAL;
    // buffers that do not hold the plan (an update that ran out of memory) launch nothing
    if (!p->host_buf || !p->dev_buf || !p->ws_o || !p->ws_lse || p->plan.items.size() > p->buf_cap_items ||
        static_cast<size_t>(std::max(p->plan.ws_slots, 0)) > p->ws_cap_slots)
        return PKV_ENOMEM;

    const int32_t* plan_buf = p->dev_buf;
    if (p->dirty && !dp && src == PlanSource::kInPlace && p->host_buf_dev) {
        plan_buf = p->host_buf_dev;
    } else if (p->dirty && !dp) {
        PKV_CUDA(cudaMemcpyAsync(p->dev_buf, p->host_buf, p->upload_bytes, cudaMemcpyHostToDevice, s));
        PKV_CUDA(cudaEventRecord(p->upload_done, s));
        p->upload_recorded = true;
        p->dirty = false;
    }
    if (k_pages != p->map_k) {
        int rc = encode_pool_map(&p->kmap, k_pages, p->g, p->page_size);
        if (rc) return rc;
        p->map_k = k_pages;
    }
    if (v_pages != p->map_v) {
        int rc = encode_pool_map(&p->vmap, v_pages, p->g, p->page_size);
        if (rc) return rc;
        p->map_v = v_pages;
    }

    const Plan& pl = p->plan;
    pkv::AttnParams a{};
    a.q = static_cast<const uint16_t*>(q);
    a.block_table = block_table_d;
    a.seq_lens = seq_lens_d;
    a.queue = reinterpret_cast<const pkv_work_item*>(plan_buf);
    a.row_start = plan_buf + p->buf_cap_items * 5;
    a.row_splits = a.row_start + p->g.batch;
    a.order = pl.mode == PKV_MODE_PERSISTENT ? a.row_splits + p->g.batch : nullptr;
    a.tiles_d = nullptr;
    a.out = out;
    a.lse = lse;
    a.ws_o = p->ws_o;
    a.ws_lse = p->ws_lse;
    a.arrive = p->arrive;
    a.ctr = p->ctr;
    a.B = p->g.batch;
    a.Hq = p->g.num_q_heads;
    a.Hkv = p->g.num_kv_heads;
    a.D = p->g.head_dim;
    a.page_size = p->page_size;
    a.max_pages = p->g.max_pages_per_seq;
    a.num_pages = p->g.num_pages;
    a.chunk_pages = pl.chunk;
    a.max_splits = pl.s_max;
    a.num_tiles = static_cast<int32_t>(pl.items.size());
    a.fused_merge = p->opts.separate_merge ? 0 : 1;
    a.all_merge = pl.merge == PKV_MERGE_ALL ? 1 : 0;
    a.use_mma = p->opts.math != PKV_MATH_FMA;
    a.copy_lsu = resolved_copy(p->opts, pl.mode) == PKV_COPY_LSU ? 1 : 0;
    a.queue_host_staged = dp || src == PlanSource::kKernelCopied ? 0 : 1;
    a.no_empty_rows = !dp && !pl.any_empty_row ? 1 : 0;
    a.k_pages = static_cast<const uint16_t*>(k_pages);
    a.v_pages = static_cast<const uint16_t*>(v_pages);
    a.scale_log2 = static_cast<float>(1.4426950408889634 / sqrt(static_cast<double>(p->g.head_dim)));
    switch (pl.mode) {
        case PKV_MODE_DIRECT: a.route = pkv::kRouteDirect; break;
        case PKV_MODE_SPLIT_QUEUE: a.route = pkv::kRouteQueue; break;
        case PKV_MODE_SPLIT_PADDED: a.route = pkv::kRoutePadded; break;
        default: a.route = pkv::kRoutePersistent; break;
    }
    int grid = pl.grid;
    bool need_merge = pl.need_merge;
    if (dp) {   // persistent route over a device-built plan; the grid is the full SM-sized one
        a.route = pkv::kRoutePersistent;
        a.queue = dp->queue;
        a.row_start = dp->row_start;
        a.row_splits = dp->row_splits;
        a.order = dp->order;
        a.tiles_d = dp->tiles;
        a.chunk_pages = dp->chunk;
        a.max_splits = dp->max_splits;
        a.fused_merge = 1;
        a.all_merge = 0;
        grid = p->num_sms * std::max(1, p->ctas_per_sm);
        need_merge = false;
    }
    *a_out = a;
    *grid_out = grid;
    *need_merge_out = need_merge;
    return PKV_OK;
}

int enqueue_decode(pkv_plan_t p, const void* q, const void* k_pages, const void* v_pages,
                   const int32_t* block_table_d, const int32_t* seq_lens_d, float* out, float* lse, cudaStream_t s,
                   const DevicePlan* dp, PlanSource src = PlanSource::kUpload) {
    if (p->g.batch == 0) return PKV_OK;
    pkv::AttnParams a{};
    int grid = 0;
    bool need_merge = false;
    int rc = prepare_decode(p, q, k_pages, v_pages, block_table_d, seq_lens_d, out, lse, s, dp, &a, &grid, &need_merge,
                            src);
    if (rc) return rc;

    if (p->profile) {
        for (auto& ev : p->ev)
            if (!ev) PKV_CUDA(cudaEventCreate(&ev));
        PKV_CUDA(cudaEventRecord(p->ev[0], s));
    }
    if (p->trace_on && grid > 0) {
        if (grid > p->trace_cap) {   // tracing is a diagnostic: its buffer grows here, synchronously
            PKV_CUDA(cudaStreamSynchronize(s));
            cudaFree(p->trace);
            p->trace = nullptr;
            p->trace_cap = 0;
            PKV_CUDA(cudaMalloc(&p->trace, static_cast<size_t>(grid) * pkv::kTraceWords * sizeof(uint64_t)));
            p->trace_cap = grid;
        }
        a.trace = p->trace;
        p->trace_rows = grid;
    }
    int n = 0;
    if (grid > 0) {
        cudaError_t e = pkv::launch_attention(a, p->kmap, p->vmap, grid, s, a.all_merge != 0);
        if (e == cudaErrorCooperativeLaunchTooLarge && a.all_merge) {
            // the device holds fewer CTAs right now than planned for: the last
            // arriving split merges instead (the counters are untouched)
            (void)cudaGetLastError();
            a.all_merge = 0;
            e = pkv::launch_attention(a, p->kmap, p->vmap, grid, s, false);
        }
        PKV_CUDA(e);
        ++n;
        if (p->profile) PKV_CUDA(cudaEventRecord(p->ev[n], s));
    }
    if (need_merge) {
        PKV_CUDA(pkv::launch_merge(a, s));
        ++n;
        if (p->profile) PKV_CUDA(cudaEventRecord(p->ev[n], s));
    }
    p->ev_launches = n;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_decode(const void* q, const void* k_pages, const void* v_pages, const int32_t* block_table_d,
               const int32_t* seq_lens_d, pkv_plan_t p, float* out, float* lse, pkv_stream_t stream) {
    NvtxRange range("pkv_decode");
    if (!p) return PKV_EINVAL;
    return enqueue_decode(p, q, k_pages, v_pages, block_table_d, seq_lens_d, out, lse,
                          reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int pkv_decode_host(const void* q_h, const void* k_pages, const void* v_pages, const int32_t* block_table_d,
                    const int32_t* seq_lens_d, pkv_plan_t p, float* out_h, float* lse_h, pkv_stream_t stream) {
    NvtxRange range("pkv_decode_host");
    if (!p) return PKV_EINVAL;
    if (p->g.batch == 0) return PKV_OK;
    if (!q_h || !out_h || !lse_h) return PKV_EINVAL;
    const size_t rows = static_cast<size_t>(p->g.batch) * p->g.num_q_heads;
    const size_t q_bytes = rows * p->g.head_dim * 2, out_bytes = rows * p->g.head_dim * 4, lse_bytes = rows * 4;
    // Pinned host buffers are in the GPU's address space (read and written
    // over NVLink-C2C on GB300): the kernel uses them in place.  Pageable ones
    // go through the plan's pinned, mapped staging with a host memcpy.
    const void* q_d = mapped_host_address(q_h, 16);
    float* out_d = static_cast<float*>(const_cast<void*>(mapped_host_address(out_h, 16)));
    float* lse_d = static_cast<float*>(const_cast<void*>(mapped_host_address(lse_h, 4)));
    const size_t off_out = round_up(q_bytes, 256), off_lse = off_out + round_up(out_bytes, 256);
    if ((!q_d || !out_d || !lse_d) && !p->host_stage) {
        void* h = nullptr;
        void* d = nullptr;
        if (cudaMallocHost(&h, off_lse + lse_bytes) != cudaSuccess) return PKV_ENOMEM;
        if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
            cudaFreeHost(h);
            return cuda_fail(cudaErrorInvalidValue);
        }
        p->host_stage = static_cast<uint8_t*>(h);
        p->host_stage_dev = static_cast<uint8_t*>(d);
    }
    if (!q_d) {
        memcpy(p->host_stage, q_h, q_bytes);
        q_d = p->host_stage_dev;
    }
    const bool stage_out = !out_d, stage_lse = !lse_d;
    if (stage_out) out_d = reinterpret_cast<float*>(p->host_stage_dev + off_out);
    if (stage_lse) lse_d = reinterpret_cast<float*>(p->host_stage_dev + off_lse);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int rc = enqueue_decode(p, q_d, k_pages, v_pages, block_table_d, seq_lens_d, out_d, lse_d, s, nullptr,
                                  PlanSource::kInPlace);
    // synchronise even after an error: a launched kernel may still read the
    // staging and the plan in host memory
    const cudaError_t e = cudaStreamSynchronize(s);
    if (rc) return rc;
    PKV_CUDA(e);
    if (stage_out) memcpy(out_h, p->host_stage + off_out, out_bytes);
    if (stage_lse) memcpy(lse_h, p->host_stage + off_lse, lse_bytes);
    return PKV_OK;
}

int pkv_append(const void* k_new, const void* v_new, void* k_pages, void* v_pages, const int32_t* block_table_d,
               int32_t* seq_lens_d, pkv_plan_t p, pkv_stream_t stream) {
    NvtxRange range("pkv_append");
    if (!p) return PKV_EINVAL;
    if (p->g.batch == 0) return PKV_OK;
    if (!k_new || !v_new || !k_pages || !v_pages || !block_table_d || !seq_lens_d) return PKV_EINVAL;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) || !aligned16(v_pages)) return PKV_EINVAL;
    PKV_CUDA(pkv::launch_append(static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
                                static_cast<uint16_t*>(k_pages), static_cast<uint16_t*>(v_pages), block_table_d,
                                seq_lens_d, p->g.batch, p->g.num_kv_heads, p->g.head_dim, p->page_size,
                                p->g.max_pages_per_seq, p->g.num_pages, &p->ctr->status,
                                reinterpret_cast<cudaStream_t>(stream)));
    return PKV_OK;
}

int pkv_status(pkv_plan_t p, pkv_stream_t stream, uint32_t* status) {
    if (!p || !status) return PKV_EINVAL;
    PKV_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    PKV_CUDA(cudaMemcpy(status, &p->ctr->status, sizeof(uint32_t), cudaMemcpyDeviceToHost));
    PKV_CUDA(cudaMemset(&p->ctr->status, 0, sizeof(uint32_t)));
    return PKV_OK;
}

int pkv_read_workspace(pkv_plan_t p, pkv_stream_t stream, float* o_h, float* lse_h, int32_t capacity,
                       int32_t* count) {
    if (!p || !count) return PKV_EINVAL;
    const int32_t n = p->plan.ws_slots;
    *count = n;
    if (!o_h || !lse_h || capacity <= 0 || n == 0) return PKV_OK;
    const int32_t m = std::min(n, capacity);
    const int G = p->g.num_q_heads / p->g.num_kv_heads;
    PKV_CUDA(cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)));
    PKV_CUDA(cudaMemcpy(o_h, p->ws_o, sizeof(float) * m * G * p->g.head_dim, cudaMemcpyDeviceToHost));
    PKV_CUDA(cudaMemcpy(lse_h, p->ws_lse, sizeof(float) * m * G, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < static_cast<int64_t>(m) * G; ++i) lse_h[i] *= 0.69314718055994530942f;
    return PKV_OK;
}

int pkv_selftest_wait(int64_t limit_ns, uint32_t* status_h, int32_t* result_h) {
    if (limit_ns <= 0 || limit_ns > 2000000000 || !status_h || !result_h) return PKV_EINVAL;
    uint32_t* status = nullptr;
    int* result = nullptr;
    if (cudaMalloc(&status, sizeof(uint32_t)) != cudaSuccess) return PKV_ENOMEM;
    if (cudaMalloc(&result, 3 * sizeof(int)) != cudaSuccess) {
        cudaFree(status);
        return PKV_ENOMEM;
    }
    cudaError_t e = cudaMemset(status, 0, sizeof(uint32_t));
    if (e == cudaSuccess) e = pkv::launch_wait_selftest(status, static_cast<uint64_t>(limit_ns), result, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(status_h, status, sizeof(uint32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemcpy(result_h, result, 3 * sizeof(int), cudaMemcpyDeviceToHost);
    cudaFree(status);
    cudaFree(result);
    return e == cudaSuccess ? PKV_OK : cuda_fail(e);
}

int pkv_profile_enable(pkv_plan_t p, int32_t enable) {
    if (!p) return PKV_EINVAL;
    p->profile = enable != 0;
    return PKV_OK;
}

int pkv_trace_enable(pkv_plan_t p, int32_t enable) {
    if (!p) return PKV_EINVAL;
    p->trace_on = enable != 0;
    return PKV_OK;
}

int pkv_trace_read(pkv_plan_t p, uint64_t* rows_h, int32_t capacity, int32_t* count) {
    if (!p || !count) return PKV_EINVAL;
    *count = p->trace ? p->trace_rows : 0;
    if (!*count || !rows_h) return PKV_OK;
    PKV_CUDA(cudaDeviceSynchronize());
    const int n = std::min(*count, std::max(capacity, 0));
    if (n > 0)
        PKV_CUDA(cudaMemcpy(rows_h, p->trace, static_cast<size_t>(n) * pkv::kTraceWords * sizeof(uint64_t),
                            cudaMemcpyDeviceToHost));
    return PKV_OK;
}

int pkv_profile_read(pkv_plan_t p, float* ms, int32_t capacity, int32_t* count) {
    if (!p || !count) return PKV_EINVAL;
    *count = p->profile ? p->ev_launches : 0;
    if (!p->profile || !ms) return PKV_OK;
    for (int i = 0; i < p->ev_launches && i < capacity; ++i) {
        PKV_CUDA(cudaEventSynchronize(p->ev[i + 1]));
        PKV_CUDA(cudaEventElapsedTime(&ms[i], p->ev[i], p->ev[i + 1]));
    }
    return PKV_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ page pool

struct pkv_pool_s {
    std::deque<int32_t> free_list;
    std::vector<uint8_t> is_free;   // [num_pages]: the page is in free_list
    int32_t num_pages = 0;
};

extern "C" {

int pkv_pool_create(const int32_t* free_pages, int32_t count, int32_t num_pages, pkv_pool_t* pool) {
    if (!pool || count < 0 || (count > 0 && !free_pages) || num_pages <= 0) return PKV_EINVAL;
    *pool = nullptr;
    for (int32_t i = 0; i < count; ++i)
        if (free_pages[i] < 0 || free_pages[i] >= num_pages) return PKV_EINVAL;
    pkv_pool_s* p = new (std::nothrow) pkv_pool_s;
    if (!p) return PKV_ENOMEM;
    p->is_free.assign(num_pages, 0);
    for (int32_t i = 0; i < count; ++i) {
        if (p->is_free[free_pages[i]]) {   // listed twice
            delete p;
            return PKV_EINVAL;
        }
        p->is_free[free_pages[i]] = 1;
    }
    p->free_list.assign(free_pages, free_pages + count);
    p->num_pages = num_pages;
    *pool = p;
    return PKV_OK;
}

}  // extern "C"

namespace {
// pkv_pool_reserve over the rows whose `active` entry is non-zero (all rows
// when `active` is null): idle slots of a session take no page.
int pool_reserve_rows(pkv_pool_t pool, const int32_t* seq_lens_h, int32_t* block_table_h, int32_t batch,
                      int32_t max_pages_per_seq, int32_t page_size, const uint8_t* active, int32_t* rows_out,
                      int32_t* n_rows) {
    if (!pool || batch < 0 || (batch > 0 && (!seq_lens_h || !block_table_h)) || max_pages_per_seq <= 0 ||
        page_size <= 0)
        return PKV_EINVAL;
    // first pass: count and check, so that failure changes nothing
    auto wants_page = [&](int32_t b) {
        return (!active || active[b]) && seq_lens_h[b] % page_size == 0 &&
               block_table_h[static_cast<size_t>(b) * max_pages_per_seq + seq_lens_h[b] / page_size] < 0;
    };
    int32_t need = 0;
    for (int32_t b = 0; b < batch; ++b) {
        if (seq_lens_h[b] < 0) return PKV_EINVAL;
        if ((!active || active[b]) && seq_lens_h[b] % page_size == 0 &&
            seq_lens_h[b] / page_size >= max_pages_per_seq)
            return PKV_ENOSPACE;
        if (wants_page(b)) ++need;
    }
    if (static_cast<size_t>(need) > pool->free_list.size()) return PKV_ENOSPACE;
    int32_t k = 0;
    for (int32_t b = 0; b < batch; ++b) {
        if (!wants_page(b)) continue;
        const int32_t page = pool->free_list.front();
        block_table_h[static_cast<size_t>(b) * max_pages_per_seq + seq_lens_h[b] / page_size] = page;
        pool->free_list.pop_front();
        pool->is_free[page] = 0;
        if (rows_out) rows_out[k] = b;
        ++k;
    }
    if (n_rows) *n_rows = k;
    return PKV_OK;
}
}  // namespace

extern "C" {

int pkv_pool_reserve(pkv_pool_t pool, const int32_t* seq_lens_h, int32_t* block_table_h, int32_t batch,
                     int32_t max_pages_per_seq, int32_t page_size, int32_t* rows_out, int32_t* n_rows) {
    return pool_reserve_rows(pool, seq_lens_h, block_table_h, batch, max_pages_per_seq, page_size, nullptr, rows_out,
                             n_rows);
}

int pkv_pool_release(pkv_pool_t pool, const int32_t* pages, int32_t count) {
    if (!pool || count < 0 || (count > 0 && !pages)) return PKV_EINVAL;
    for (int32_t i = 0; i < count; ++i)
        if (pages[i] < 0 || pages[i] >= pool->num_pages) return PKV_EINVAL;
    // a page that is free already (or listed twice) is refused, and nothing changes
    for (int32_t i = 0; i < count; ++i) {
        if (pool->is_free[pages[i]]) {
            for (int32_t j = 0; j < i; ++j) pool->is_free[pages[j]] = 0;
            return PKV_EINVAL;
        }
        pool->is_free[pages[i]] = 1;
    }
    pool->free_list.insert(pool->free_list.end(), pages, pages + count);
    return PKV_OK;
}

int32_t pkv_pool_free_count(pkv_pool_t pool) { return pool ? static_cast<int32_t>(pool->free_list.size()) : 0; }

void pkv_pool_destroy(pkv_pool_t pool) { delete pool; }

}  // extern "C"

// ------------------------------------------------------------------ continuous sessions
//
// A cohort of rows that each grow by one token per step, advanced together as
// the resident program of "WPK persistent kernel" (dotwave.ai) advances its
// sessions each beat.  One step: the pool hands a page to every row whose next
// token starts one (only those table entries travel to the device), the plan
// is rebuilt for the lengths after the append, then append and decode are
// enqueued back to back.  Host mirrors of lengths and table live in pinned
// memory; the device table and lengths belong to the caller.

struct pkv_session_s {
    pkv_plan_t plan = nullptr;
    pkv_pool_t pool = nullptr;
    int32_t* lens_h = nullptr;    // pinned [B]
    int32_t* table_h = nullptr;   // pinned [B][max_pages]
    int32_t* rows = nullptr;      // [B] scratch for the pool's touched rows
    int32_t* table_d = nullptr;
    int32_t* lens_d = nullptr;
    cudaEvent_t copied = nullptr;   // the last step's table entries (and new_pages) have been read
    bool copy_pending = false;
    // host-planned steps: per row (table index, page id) of the step's new page,
    // pinned and mapped; read by the step's append kernel (index -1: none)
    int32_t* new_pages_h = nullptr;
    const int32_t* new_pages_d = nullptr;
    // device-planned steps (pkv_session_device_plan)
    bool device_mode = false;
    int32_t* dev_free = nullptr;        // free page ids, handed out in order
    uint32_t* dev_free_state = nullptr; // {next index, pages left}
    int32_t free_cap = 0;
    int32_t* dev_plan = nullptr;        // [queue_cap * 5][B][B][queue_cap][1]
    int32_t queue_cap = 0;
    int32_t chunk = 0;
    int32_t max_splits = 0;
    pkv_resident_s* resident = nullptr;   // a resident kernel owns the session's device state
    // slots: active rows take a token each step, idle ones (evicted) are left alone
    int32_t* active_d = nullptr;             // [B] device, 1 active / 0 idle
    std::vector<uint8_t> active_h;            // the host's view of the same
    pkv::SlotRequest* req_h = nullptr;        // pinned, mapped [B] slot requests of one call
    const pkv::SlotRequest* req_d = nullptr;
    int32_t* req_pages_h = nullptr;           // pinned, mapped page ids chosen by the host pool
    const int32_t* req_pages_d = nullptr;
    size_t req_pages_cap = 0;
};

struct pkv_resident_s {
    pkv_session_t session = nullptr;
    cudaStream_t kstream = nullptr;   // the resident kernel (non-blocking)
    cudaStream_t cstream = nullptr;   // the per-step copies (non-blocking)
    pkv::ResidentCtl* ctl_h = nullptr;   // mapped pinned control block
    pkv::ResidentCtl* ctl_d = nullptr;
    uint32_t* grid_sync = nullptr;
    uint64_t* times_d = nullptr;
    int32_t times_cap = 0;
    void* q_d = nullptr;
    void* k_new_d = nullptr;
    void* v_new_d = nullptr;
    float* out_d = nullptr;
    float* lse_d = nullptr;
    size_t q_bytes = 0, new_bytes = 0, out_bytes = 0, lse_bytes = 0;
    uint32_t step = 0;
    bool running = false;
    pkv::SlotRequest* req_h = nullptr;   // pinned, mapped slot requests for the next step
    const pkv::SlotRequest* req_d = nullptr;
    int32_t n_req = 0;
    uint32_t* row_ready = nullptr;       // device [B]: the last step whose append of the row landed
    pkv::ResidentParams rp{};            // the launch's parameters (relaunched after a yield)
    int grid = 0;
    int32_t yield_every = 0;
    uint32_t launch_first = 1;           // the first step of the current launch
    bool yielded = false;                // the kernel left the GPU after yield_every steps
    int32_t launches = 0;
};

namespace {
void session_free(pkv_session_s* s) {
    if (!s) return;
    if (s->copy_pending) cudaEventSynchronize(s->copied);
    cudaFree(s->dev_free);
    cudaFree(s->dev_free_state);
    cudaFree(s->dev_plan);
    cudaFree(s->active_d);
    cudaFreeHost(s->req_h);
    cudaFreeHost(s->req_pages_h);
    cudaFreeHost(s->lens_h);
    cudaFreeHost(s->table_h);
    cudaFreeHost(s->new_pages_h);
    delete[] s->rows;
    if (s->copied) cudaEventDestroy(s->copied);
    delete s;
}
}  // namespace

extern "C" {

int pkv_session_create(pkv_plan_t plan, pkv_pool_t pool, const int32_t* seq_lens_h, const int32_t* block_table_h,
                       int32_t* block_table_d, int32_t* seq_lens_d, pkv_session_t* session) {
    if (!session) return PKV_EINVAL;
    *session = nullptr;
    if (!plan || !pool || !block_table_d || !seq_lens_d || (plan->g.batch > 0 && (!seq_lens_h || !block_table_h)))
        return PKV_EINVAL;
    const int B = plan->g.batch;
    const size_t table_n = static_cast<size_t>(B) * plan->g.max_pages_per_seq;
    int rc = validate_rows(plan->g, plan->page_size, seq_lens_h, block_table_h);
    if (rc) return rc;
    pkv_session_s* s = new (std::nothrow) pkv_session_s;
    if (!s) return PKV_ENOMEM;
    s->plan = plan;
    s->pool = pool;
    s->table_d = block_table_d;
    s->lens_d = seq_lens_d;
    s->rows = new (std::nothrow) int32_t[std::max(B, 1)];
    if (!s->rows || cudaMallocHost(&s->lens_h, sizeof(int32_t) * std::max(B, 1)) != cudaSuccess ||
        cudaMallocHost(&s->table_h, sizeof(int32_t) * std::max<size_t>(table_n, 1)) != cudaSuccess ||
        cudaMallocHost(&s->new_pages_h, sizeof(int32_t) * 2 * std::max(B, 1)) != cudaSuccess ||
        cudaEventCreateWithFlags(&s->copied, cudaEventDisableTiming) != cudaSuccess) {
        session_free(s);
        return PKV_ENOMEM;
    }
    void* mapped = nullptr;
    if (cudaHostGetDevicePointer(&mapped, s->new_pages_h, 0) == cudaSuccess)
        s->new_pages_d = static_cast<const int32_t*>(mapped);
    else
        (void)cudaGetLastError();   // not mapped: steps copy table entries with the copy engine
    if (B > 0) {
        memcpy(s->lens_h, seq_lens_h, sizeof(int32_t) * B);
        memcpy(s->table_h, block_table_h, sizeof(int32_t) * table_n);
    }
    // every row starts active
    s->active_h.assign(B, 1);
    const std::vector<int32_t> ones(std::max(B, 1), 1);
    if (cudaMalloc(&s->active_d, sizeof(int32_t) * std::max(B, 1)) != cudaSuccess ||
        cudaHostAlloc(&s->req_h, sizeof(pkv::SlotRequest) * std::max(B, 1), cudaHostAllocMapped) != cudaSuccess) {
        session_free(s);
        return PKV_ENOMEM;
    }
    cudaError_t e = cudaMemcpy(s->active_d, ones.data(), sizeof(int32_t) * std::max(B, 1), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(&mapped, s->req_h, 0);
    if (e != cudaSuccess) {
        session_free(s);
        return cuda_fail(e);
    }
    s->req_d = static_cast<const pkv::SlotRequest*>(mapped);
    *session = s;
    return PKV_OK;
}

int pkv_session_device_plan(pkv_session_t s, pkv_stream_t stream) {
    NvtxRange range("pkv_session_device_plan");
    if (!s) return PKV_EINVAL;
    if (s->device_mode) return PKV_OK;
    pkv_plan_s* p = s->plan;
    const pkv_geom& g = p->g;
    const int B = g.batch, Hkv = g.num_kv_heads, G = g.num_q_heads / g.num_kv_heads;
    if (p->plan.mode != PKV_MODE_PERSISTENT || B > pkv::kDevPlanMaxRows) return PKV_EUNSUPPORTED;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (s->copy_pending) {
        PKV_CUDA(cudaEventSynchronize(s->copied));
        s->copy_pending = false;
    }
    // one split per row stays one split however long the rows grow
    const int32_t chunk = p->opts.num_splits == 1 ? g.max_pages_per_seq : p->plan.chunk;
    const int32_t s_max = static_cast<int32_t>(ceil_div(g.max_pages_per_seq, chunk));
    if (static_cast<int64_t>(s_max) * G > pkv::kMergeCapFloats) return PKV_EUNSUPPORTED;
    const int64_t cap = static_cast<int64_t>(B) * Hkv * s_max;
    if (cap > INT32_MAX / 8) return PKV_EUNSUPPORTED;
    // workspace for the largest plan the table allows
    if (static_cast<size_t>(cap) > p->ws_cap_slots) {
        cudaFree(p->ws_o);
        cudaFree(p->ws_lse);
        p->ws_o = nullptr;
        p->ws_lse = nullptr;
        p->ws_cap_slots = 0;
        if (cudaMalloc(&p->ws_o, cap * G * g.head_dim * sizeof(float)) != cudaSuccess) return PKV_ENOMEM;
        if (cudaMalloc(&p->ws_lse, cap * G * sizeof(float)) != cudaSuccess) return PKV_ENOMEM;
        p->ws_cap_slots = cap;
    }
    std::vector<int32_t> pages(s->pool->free_list.begin(), s->pool->free_list.end());
    const size_t plan_ints = static_cast<size_t>(cap) * 6 + 2 * static_cast<size_t>(B) + 1;
    // the free list is a ring that can hold every page of the pool (evicted rows give theirs back)
    const size_t ring = std::max<size_t>(std::max<size_t>(pages.size(), static_cast<size_t>(g.num_pages)), 1);
    if (cudaMalloc(&s->dev_plan, plan_ints * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&s->dev_free, ring * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&s->dev_free_state, 2 * sizeof(uint32_t)) != cudaSuccess) {
        cudaFree(s->dev_plan);   // none of them is kept: a later call starts over
        cudaFree(s->dev_free);
        cudaFree(s->dev_free_state);
        s->dev_plan = nullptr;
        s->dev_free = nullptr;
        s->dev_free_state = nullptr;
        return PKV_ENOMEM;
    }
    const uint32_t state[2] = {0u, static_cast<uint32_t>(pages.size())};
    PKV_CUDA(cudaMemcpyAsync(s->dev_free, pages.data(), pages.size() * sizeof(int32_t), cudaMemcpyHostToDevice, st));
    PKV_CUDA(cudaMemcpyAsync(s->dev_free_state, state, sizeof(state), cudaMemcpyHostToDevice, st));
    PKV_CUDA(cudaStreamSynchronize(st));   // the host vectors above go out of scope
    s->pool->free_list.clear();            // those pages now belong to the device allocator
    std::fill(s->pool->is_free.begin(), s->pool->is_free.end(), uint8_t{0});
    s->free_cap = static_cast<int32_t>(ring);
    s->queue_cap = static_cast<int32_t>(cap);
    s->chunk = chunk;
    s->max_splits = s_max;
    s->device_mode = true;
    return PKV_OK;
}

namespace {
// The device planner's parameters and the decode's view of the device plan.
void device_plan_views(pkv_session_t s, pkv::DevPlanParams* dp_out, DevicePlan* plan_out) {
    pkv_plan_s* p = s->plan;
    const pkv_geom& g = p->g;
    const int B = g.batch;
    int32_t* q_items = s->dev_plan;
    int32_t* row_start = q_items + static_cast<size_t>(s->queue_cap) * 5;
    int32_t* row_splits = row_start + B;
    int32_t* order = row_splits + B;
    int32_t* tiles = order + s->queue_cap;
    pkv::DevPlanParams dp{};
    dp.lens = s->lens_d;
    dp.active = s->active_d;
    dp.table = s->table_d;
    dp.free_list = s->dev_free;
    dp.free_state = s->dev_free_state;
    dp.free_cap = s->free_cap;
    dp.queue = reinterpret_cast<pkv_work_item*>(q_items);
    dp.row_start = row_start;
    dp.row_splits = row_splits;
    dp.order = order;
    dp.tiles = tiles;
    dp.queue_cap = s->queue_cap;
    dp.status = &p->ctr->status;
    dp.B = B;
    dp.Hkv = g.num_kv_heads;
    dp.page_size = p->page_size;
    dp.max_pages = g.max_pages_per_seq;
    dp.chunk = s->chunk;
    *dp_out = dp;
    *plan_out = DevicePlan{reinterpret_cast<const pkv_work_item*>(q_items), row_start, row_splits, order, tiles,
                           s->chunk, s->max_splits};
}

int session_step_device(pkv_session_t s, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                        const void* q, float* out, float* lse, cudaStream_t st) {
    pkv_plan_s* p = s->plan;
    pkv::DevPlanParams dp{};
    DevicePlan plan{};
    device_plan_views(s, &dp, &plan);
    if (!k_new || !v_new || !k_pages || !v_pages || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pages) ||
        !aligned16(v_pages))
        return PKV_EINVAL;
    PKV_CUDA(pkv::launch_plan_step(dp, st));
    const pkv_geom& g = p->g;
    PKV_CUDA(pkv::launch_append(static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
                                static_cast<uint16_t*>(k_pages), static_cast<uint16_t*>(v_pages), s->table_d,
                                s->lens_d, g.batch, g.num_kv_heads, g.head_dim, p->page_size, g.max_pages_per_seq,
                                g.num_pages, &p->ctr->status, st, s->active_d));
    return enqueue_decode(p, q, k_pages, v_pages, s->table_d, s->lens_d, out, lse, st, &plan);
}
}  // namespace

int pkv_session_step(pkv_session_t s, const void* k_new, const void* v_new, void* k_pages, void* v_pages,
                     const void* q, float* out, float* lse, pkv_stream_t stream) {
    NvtxRange range("pkv_session_step");
    if (!s || s->resident) return PKV_EINVAL;
    const pkv_geom& g = s->plan->g;
    const int B = g.batch, ps = s->plan->page_size, mp = g.max_pages_per_seq;
    if (B == 0) return PKV_OK;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (s->device_mode) return session_step_device(s, k_new, v_new, k_pages, v_pages, q, out, lse, st);
    // every pointer is checked before the step changes any state
    if (!k_new || !v_new || !k_pages || !v_pages || !q || !out || !lse || !aligned16(k_new) || !aligned16(v_new) ||
        !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(q) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return PKV_EINVAL;
    if (s->copy_pending) {
        PKV_CUDA(cudaEventSynchronize(s->copied));
        s->copy_pending = false;
    }
    int32_t n_rows = 0;
    int rc = pool_reserve_rows(s->pool, s->lens_h, s->table_h, B, mp, ps, s->active_h.data(), s->rows, &n_rows);
    if (rc) return rc;
    pkv_plan_s* p = s->plan;
    if (s->new_pages_d && p->host_buf_dev) {
        // One launch does the step's host -> device traffic: it enters the new pages
        // in the table, copies the re-planned queue into the plan's device buffer and
        // appends the tokens; then the decode.  No copy engine is used.
        for (int b = 0; b < B; ++b) s->new_pages_h[2 * b] = -1;
        for (int32_t i = 0; i < n_rows; ++i) {
            const int b = s->rows[i];
            s->new_pages_h[2 * b] = s->lens_h[b] / ps;
            s->new_pages_h[2 * b + 1] = s->table_h[static_cast<size_t>(b) * mp + s->lens_h[b] / ps];
        }
        for (int b = 0; b < B; ++b) s->lens_h[b] += s->active_h[b];   // idle slots do not grow
        if ((rc = pkv_plan_update(p, s->lens_h, nullptr))) return rc;
        pkv::AppendStepParams ap{};
        ap.k_new = static_cast<const uint16_t*>(k_new);
        ap.v_new = static_cast<const uint16_t*>(v_new);
        ap.k_pages = static_cast<uint16_t*>(k_pages);
        ap.v_pages = static_cast<uint16_t*>(v_pages);
        ap.block_table = s->table_d;
        ap.seq_lens = s->lens_d;
        ap.new_pages = s->new_pages_d;
        ap.active = s->active_d;
        // (a plan staging that is not mapped is uploaded by the decode's copy instead)
        const bool kernel_copies = p->dirty && p->host_buf_dev;
        if (kernel_copies) {
            ap.plan_src = p->host_buf_dev;
            ap.plan_dst = p->dev_buf;
            ap.plan_words = static_cast<int64_t>(p->upload_bytes / sizeof(int32_t));
        }
        ap.status = &p->ctr->status;
        ap.B = B;
        ap.Hkv = g.num_kv_heads;
        ap.D = g.head_dim;
        ap.page_size = ps;
        ap.max_pages = mp;
        ap.num_pages = g.num_pages;
        PKV_CUDA(pkv::launch_append_step(ap, st));
        // the host staging (plan, new pages) may be rewritten once this kernel is done
        PKV_CUDA(cudaEventRecord(s->copied, st));
        s->copy_pending = true;
        if (kernel_copies) {
            PKV_CUDA(cudaEventRecord(p->upload_done, st));
            p->upload_recorded = true;
            p->dirty = false;
        }
        return enqueue_decode(p, q, k_pages, v_pages, s->table_d, s->lens_d, out, lse, st, nullptr,
                              PlanSource::kKernelCopied);
    }
    for (int32_t i = 0; i < n_rows; ++i) {
        const size_t at = static_cast<size_t>(s->rows[i]) * mp + s->lens_h[s->rows[i]] / ps;
        PKV_CUDA(cudaMemcpyAsync(s->table_d + at, s->table_h + at, sizeof(int32_t), cudaMemcpyHostToDevice, st));
    }
    if (n_rows > 0) {
        PKV_CUDA(cudaEventRecord(s->copied, st));
        s->copy_pending = true;
    }
    for (int b = 0; b < B; ++b) s->lens_h[b] += s->active_h[b];   // idle slots do not grow
    if ((rc = pkv_plan_update(s->plan, s->lens_h, nullptr))) return rc;
    PKV_CUDA(pkv::launch_append(static_cast<const uint16_t*>(k_new), static_cast<const uint16_t*>(v_new),
                                static_cast<uint16_t*>(k_pages), static_cast<uint16_t*>(v_pages), s->table_d,
                                s->lens_d, B, g.num_kv_heads, g.head_dim, ps, mp, g.num_pages, &p->ctr->status, st,
                                s->active_d));
    return pkv_decode(q, k_pages, v_pages, s->table_d, s->lens_d, s->plan, out, lse, stream);
}

int pkv_session_lengths(pkv_session_t s, int32_t* seq_lens_h) {
    if (!s || !seq_lens_h || s->resident) return PKV_EINVAL;
    const size_t bytes = sizeof(int32_t) * s->plan->g.batch;
    if (s->device_mode) {   // the device holds the truth; synchronises the device
        PKV_CUDA(cudaDeviceSynchronize());
        PKV_CUDA(cudaMemcpy(seq_lens_h, s->lens_d, bytes, cudaMemcpyDeviceToHost));
    } else {
        memcpy(seq_lens_h, s->lens_h, bytes);
    }
    return PKV_OK;
}

int pkv_session_table(pkv_session_t s, int32_t* block_table_h) {
    if (!s || !block_table_h || s->resident) return PKV_EINVAL;
    const size_t bytes = sizeof(int32_t) * static_cast<size_t>(s->plan->g.batch) * s->plan->g.max_pages_per_seq;
    if (s->device_mode) {
        PKV_CUDA(cudaDeviceSynchronize());
        PKV_CUDA(cudaMemcpy(block_table_h, s->table_d, bytes, cudaMemcpyDeviceToHost));
    } else {
        memcpy(block_table_h, s->table_h, bytes);
    }
    return PKV_OK;
}

int pkv_session_device_queue(pkv_session_t s, pkv_work_item* items, int32_t* order, int32_t capacity,
                             int32_t* count) {
    if (!s || !count || s->resident) return PKV_EINVAL;
    if (!s->device_mode) return PKV_EINVAL;
    PKV_CUDA(cudaDeviceSynchronize());
    const int32_t* tiles = s->dev_plan + static_cast<size_t>(s->queue_cap) * 6 + 2 * s->plan->g.batch;
    int32_t n = 0;
    PKV_CUDA(cudaMemcpy(&n, tiles, sizeof(int32_t), cudaMemcpyDeviceToHost));
    *count = n;
    const int32_t m = std::min(n, capacity);
    if (items && m > 0)
        PKV_CUDA(cudaMemcpy(items, s->dev_plan, sizeof(pkv_work_item) * m, cudaMemcpyDeviceToHost));
    if (order && m > 0)
        PKV_CUDA(cudaMemcpy(order, s->dev_plan + static_cast<size_t>(s->queue_cap) * 5 + 2 * s->plan->g.batch,
                            sizeof(int32_t) * m, cudaMemcpyDeviceToHost));
    return PKV_OK;
}

// ------------------------------------------------------------------ slot admit / evict
//
// A session's rows are fixed slots, reset at a step boundary as the per-session
// arenas of "WPK persistent kernel" (dotwave.ai, "What has to exist instead")
// are.  The host pool's bookkeeping runs here; with a device free list
// (device-plan mode) the slot kernel does it (pkv_slots.cuh).

namespace {

// Checks shared by the session and resident calls: rows in range, not listed
// twice, in the state the request needs (`want_active`: evictions need an
// active row, admissions an idle one); lengths fit the table; prompt pointers.
int check_slot_rows(const std::vector<uint8_t>& active, int B, const int32_t* rows_h, int32_t n, bool want_active) {
    if (n < 0 || (n > 0 && !rows_h)) return PKV_EINVAL;
    std::vector<uint8_t> seen(B, 0);
    for (int32_t i = 0; i < n; ++i) {
        const int32_t b = rows_h[i];
        if (b < 0 || b >= B || seen[b] || (active[b] != 0) != want_active) return PKV_EINVAL;
        seen[b] = 1;
    }
    return PKV_OK;
}

int check_admit_args(const pkv_plan_s* p, const int32_t* lens_h, int32_t n, const void* k_src, const void* v_src,
                     int64_t* tokens) {
    int64_t total = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (!lens_h || lens_h[i] < 0 ||
            static_cast<int64_t>(lens_h[i]) > static_cast<int64_t>(p->g.max_pages_per_seq) * p->page_size)
            return PKV_EINVAL;
        total += lens_h[i];
    }
    if (total > 0 && (!k_src || !v_src || !aligned16(k_src) || !aligned16(v_src))) return PKV_EINVAL;
    if (total > INT32_MAX) return PKV_EINVAL;
    *tokens = total;
    return PKV_OK;
}

pkv::SlotParams slot_params(pkv_session_t s, void* k_pages, void* v_pages, int32_t n) {
    pkv_plan_s* p = s->plan;
    pkv::SlotParams sp{};
    sp.req = s->req_d;
    sp.n = n;
    sp.pages = s->req_pages_d;
    if (s->device_mode) {
        sp.free_list = s->dev_free;
        sp.free_state = s->dev_free_state;
        sp.free_cap = s->free_cap;
    }
    sp.table = s->table_d;
    sp.lens = s->lens_d;
    sp.active = s->active_d;
    sp.k_pages = static_cast<uint16_t*>(k_pages);
    sp.v_pages = static_cast<uint16_t*>(v_pages);
    sp.status = &p->ctr->status;
    sp.B = p->g.batch;
    sp.Hkv = p->g.num_kv_heads;
    sp.D = p->g.head_dim;
    sp.page_size = p->page_size;
    sp.max_pages = p->g.max_pages_per_seq;
    sp.num_pages = p->g.num_pages;
    return sp;
}

// The staging of the last slot call (or step) may still be read by the GPU.
int wait_session_staging(pkv_session_t s) {
    if (s->copy_pending) {
        PKV_CUDA(cudaEventSynchronize(s->copied));
        s->copy_pending = false;
    }
    return PKV_OK;
}

int launch_slots(pkv_session_t s, void* k_pages, void* v_pages, int32_t n, cudaStream_t st) {
    PKV_CUDA(pkv::launch_slot_requests(slot_params(s, k_pages, v_pages, n), st));
    PKV_CUDA(cudaEventRecord(s->copied, st));   // the requests (and page ids) are read by then
    s->copy_pending = true;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_session_evict(pkv_session_t s, const int32_t* rows_h, int32_t n, pkv_stream_t stream) {
    NvtxRange range("pkv_session_evict");
    if (!s || s->resident) return PKV_EINVAL;
    const int B = s->plan->g.batch, mp = s->plan->g.max_pages_per_seq;
    int rc = check_slot_rows(s->active_h, B, rows_h, n, true);
    if (rc || n == 0) return rc;
    if ((rc = wait_session_staging(s))) return rc;
    if (!s->device_mode) {   // the host pool takes the pages back, in table order, rows in the order listed
        std::vector<int32_t> pages;
        for (int32_t i = 0; i < n; ++i)
            for (int j = 0; j < mp; ++j) {
                const int32_t page = s->table_h[static_cast<size_t>(rows_h[i]) * mp + j];
                if (page >= 0) pages.push_back(page);
            }
        if ((rc = pkv_pool_release(s->pool, pages.data(), static_cast<int32_t>(pages.size())))) return rc;
        for (int32_t i = 0; i < n; ++i) {
            std::fill(s->table_h + static_cast<size_t>(rows_h[i]) * mp,
                      s->table_h + static_cast<size_t>(rows_h[i] + 1) * mp, -1);
            s->lens_h[rows_h[i]] = 0;
        }
    }
    for (int32_t i = 0; i < n; ++i) {
        s->req_h[i] = pkv::SlotRequest{rows_h[i], -1, 0, 0, nullptr, nullptr};
        s->active_h[rows_h[i]] = 0;
    }
    return launch_slots(s, nullptr, nullptr, n, reinterpret_cast<cudaStream_t>(stream));
}

int pkv_session_admit(pkv_session_t s, const int32_t* rows_h, const int32_t* lens_h, int32_t n, const void* k_src,
                      const void* v_src, void* k_pages, void* v_pages, pkv_stream_t stream) {
    NvtxRange range("pkv_session_admit");
    if (!s || s->resident) return PKV_EINVAL;
    pkv_plan_s* p = s->plan;
    const int B = p->g.batch, mp = p->g.max_pages_per_seq, ps = p->page_size;
    int rc = check_slot_rows(s->active_h, B, rows_h, n, false);
    if (rc || n == 0) return rc;
    int64_t tokens = 0;
    if ((rc = check_admit_args(p, lens_h, n, k_src, v_src, &tokens))) return rc;
    if (!k_pages || !v_pages || !aligned16(k_pages) || !aligned16(v_pages)) return PKV_EINVAL;
    if ((rc = wait_session_staging(s))) return rc;
    int32_t src_tok = 0;
    if (!s->device_mode) {   // the host pool hands the pages out
        int64_t need = 0;
        for (int32_t i = 0; i < n; ++i) need += ceil_div(lens_h[i], ps);
        if (static_cast<size_t>(need) > s->pool->free_list.size()) return PKV_ENOSPACE;
        if (static_cast<size_t>(need) > s->req_pages_cap) {
            cudaFreeHost(s->req_pages_h);
            s->req_pages_h = nullptr;
            s->req_pages_d = nullptr;
            s->req_pages_cap = 0;
            const size_t cap = std::max<size_t>(static_cast<size_t>(need), 64);
            if (cudaHostAlloc(&s->req_pages_h, cap * sizeof(int32_t), cudaHostAllocMapped) != cudaSuccess)
                return PKV_ENOMEM;
            void* mapped = nullptr;
            PKV_CUDA(cudaHostGetDevicePointer(&mapped, s->req_pages_h, 0));
            s->req_pages_d = static_cast<const int32_t*>(mapped);
            s->req_pages_cap = cap;
        }
        int32_t off = 0;
        for (int32_t i = 0; i < n; ++i) {
            const int32_t b = rows_h[i];
            const int32_t want = static_cast<int32_t>(ceil_div(lens_h[i], ps));
            for (int32_t j = 0; j < want; ++j) {
                const int32_t page = s->pool->free_list.front();
                s->pool->free_list.pop_front();
                s->pool->is_free[page] = 0;
                s->table_h[static_cast<size_t>(b) * mp + j] = page;
                s->req_pages_h[off + j] = page;
            }
            s->lens_h[b] = lens_h[i];
            s->req_h[i] = pkv::SlotRequest{b, lens_h[i], src_tok, off, static_cast<const uint16_t*>(k_src),
                                           static_cast<const uint16_t*>(v_src)};
            off += want;
            src_tok += lens_h[i];
            s->active_h[b] = 1;
        }
    } else {   // the device free list hands them out, in the slot kernel
        for (int32_t i = 0; i < n; ++i) {
            s->req_h[i] = pkv::SlotRequest{rows_h[i], lens_h[i], src_tok, -1, static_cast<const uint16_t*>(k_src),
                                           static_cast<const uint16_t*>(v_src)};
            src_tok += lens_h[i];
            s->active_h[rows_h[i]] = 1;
        }
    }
    return launch_slots(s, k_pages, v_pages, n, reinterpret_cast<cudaStream_t>(stream));
}

int pkv_session_free_pages(pkv_session_t s, int32_t* pages_h, int32_t capacity, int32_t* count, int32_t* active_h) {
    if (!s || !count || s->resident || capacity < 0 || (capacity > 0 && !pages_h)) return PKV_EINVAL;
    const int B = s->plan->g.batch;
    if (!s->device_mode) {
        *count = static_cast<int32_t>(s->pool->free_list.size());
        int32_t i = 0;
        for (auto it = s->pool->free_list.begin(); it != s->pool->free_list.end() && i < capacity; ++it) pages_h[i++] = *it;
        if (active_h)
            for (int b = 0; b < B; ++b) active_h[b] = s->active_h[b];
        return PKV_OK;
    }
    PKV_CUDA(cudaDeviceSynchronize());
    uint32_t state[2] = {0, 0};
    PKV_CUDA(cudaMemcpy(state, s->dev_free_state, sizeof(state), cudaMemcpyDeviceToHost));
    std::vector<int32_t> ring(s->free_cap);
    PKV_CUDA(cudaMemcpy(ring.data(), s->dev_free, ring.size() * sizeof(int32_t), cudaMemcpyDeviceToHost));
    *count = static_cast<int32_t>(state[1]);
    for (uint32_t i = 0; i < state[1] && static_cast<int32_t>(i) < capacity; ++i)
        pages_h[i] = ring[(state[0] + i) % static_cast<uint32_t>(s->free_cap)];
    if (active_h && B > 0) PKV_CUDA(cudaMemcpy(active_h, s->active_d, sizeof(int32_t) * B, cudaMemcpyDeviceToHost));
    return PKV_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ resident steps

namespace {
void resident_free(pkv_resident_s* r) {
    if (!r) return;
    cudaFreeHost(r->ctl_h);
    cudaFreeHost(r->req_h);
    cudaFree(r->row_ready);
    cudaFree(r->grid_sync);
    cudaFree(r->times_d);
    if (r->kstream) cudaStreamDestroy(r->kstream);
    if (r->cstream) cudaStreamDestroy(r->cstream);
    delete r;
}

uint32_t host_load(const uint32_t* p) { return __atomic_load_n(p, __ATOMIC_ACQUIRE); }
void host_store(uint32_t* p, uint32_t v) { __atomic_store_n(p, v, __ATOMIC_SEQ_CST); }
}  // namespace

int pkv_resident_start(pkv_session_t s, void* k_pages, void* v_pages, void* q_d, void* k_new_d, void* v_new_d,
                       float* out_d, float* lse_d, int64_t idle_limit_ns, int32_t times_cap, int32_t yield_every,
                       pkv_resident_t* out) {
    NvtxRange range("pkv_resident_start");
    if (!out) return PKV_EINVAL;
    *out = nullptr;
    if (!s || !s->device_mode || s->resident || !k_pages || !v_pages || !q_d || !k_new_d || !v_new_d || !out_d ||
        !lse_d || idle_limit_ns <= 0 || idle_limit_ns > 60000000000ll || times_cap < 0 || yield_every < 0)
        return PKV_EINVAL;
    if (!aligned16(k_new_d) || !aligned16(v_new_d)) return PKV_EINVAL;
    pkv_plan_s* p = s->plan;
    const pkv_geom& g = p->g;
    if (g.batch == 0) return PKV_EINVAL;
    const int G = g.num_q_heads / g.num_kv_heads;
    int dev_sms = 0;
    PKV_CUDA(cudaDeviceGetAttribute(&dev_sms, cudaDevAttrMultiProcessorCount, p->device));
    const int per_sm = pkv::resident_ctas_per_sm(g.head_dim, G, p->opts.math != PKV_MATH_FMA);
    if (per_sm <= 0) return PKV_EUNSUPPORTED;

    pkv_resident_s* r = new (std::nothrow) pkv_resident_s;
    if (!r) return PKV_ENOMEM;
    r->session = s;
    r->q_d = q_d;
    r->k_new_d = k_new_d;
    r->v_new_d = v_new_d;
    r->out_d = out_d;
    r->lse_d = lse_d;
    r->q_bytes = static_cast<size_t>(g.batch) * g.num_q_heads * g.head_dim * 2;
    r->new_bytes = static_cast<size_t>(g.batch) * g.num_kv_heads * g.head_dim * 2;
    r->out_bytes = static_cast<size_t>(g.batch) * g.num_q_heads * g.head_dim * 4;
    r->lse_bytes = static_cast<size_t>(g.batch) * g.num_q_heads * 4;
    r->times_cap = times_cap;
    const size_t times_bytes = sizeof(uint64_t) * 4 * std::max(times_cap, 1);
    if (cudaStreamCreateWithFlags(&r->kstream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&r->cstream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaHostAlloc(&r->ctl_h, sizeof(pkv::ResidentCtl), cudaHostAllocMapped) != cudaSuccess ||
        cudaHostAlloc(&r->req_h, sizeof(pkv::SlotRequest) * PKV_RESIDENT_MAX_REQUESTS, cudaHostAllocMapped) !=
            cudaSuccess ||
        cudaMalloc(&r->grid_sync, sizeof(uint32_t) * pkv::kSyncWords) != cudaSuccess ||
        cudaMalloc(&r->row_ready, sizeof(uint32_t) * g.batch) != cudaSuccess ||
        cudaMalloc(&r->times_d, times_bytes) != cudaSuccess) {
        resident_free(r);
        return PKV_ENOMEM;
    }
    memset(r->ctl_h, 0, sizeof(pkv::ResidentCtl));
    cudaError_t e = cudaHostGetDevicePointer(reinterpret_cast<void**>(&r->ctl_d), r->ctl_h, 0);
    void* req_mapped = nullptr;
    if (e == cudaSuccess) e = cudaHostGetDevicePointer(&req_mapped, r->req_h, 0);
    r->req_d = static_cast<const pkv::SlotRequest*>(req_mapped);
    if (e == cudaSuccess) e = cudaMemset(r->grid_sync, 0, sizeof(uint32_t) * pkv::kSyncWords);
    if (e == cudaSuccess) e = cudaMemset(r->row_ready, 0, sizeof(uint32_t) * g.batch);
    if (e == cudaSuccess) e = cudaMemset(r->times_d, 0, times_bytes);
    // the kernel takes over the session's device state: earlier work on any stream must be done
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        resident_free(r);
        return cuda_fail(e);
    }

    pkv::DevPlanParams dp{};
    DevicePlan plan{};
    device_plan_views(s, &dp, &plan);
    pkv::AttnParams a{};
    int grid = 0;
    bool need_merge = false;
    int rc = prepare_decode(p, q_d, k_pages, v_pages, s->table_d, s->lens_d, out_d, lse_d, r->kstream, &plan, &a, &grid,
                            &need_merge);
    if (rc) {
        resident_free(r);
        return rc;
    }
    pkv::ResidentParams rp{};
    rp.attn = a;
    rp.plan = dp;
    rp.slots = slot_params(s, k_pages, v_pages, 0);
    rp.slots.req = r->req_d;
    rp.k_new = static_cast<const uint16_t*>(k_new_d);
    rp.v_new = static_cast<const uint16_t*>(v_new_d);
    rp.k_pages_w = static_cast<uint16_t*>(k_pages);
    rp.v_pages_w = static_cast<uint16_t*>(v_pages);
    rp.lens_w = s->lens_d;
    rp.ctl = r->ctl_d;
    rp.grid_sync = r->grid_sync;
    rp.times = times_cap > 0 ? r->times_d : nullptr;
    rp.times_cap = std::max(times_cap, 1);
    rp.idle_limit_ns = static_cast<uint64_t>(idle_limit_ns);
    rp.row_ready = r->row_ready;
    rp.first_step = 1;
    rp.yield_every = yield_every;
    r->rp = rp;
    r->grid = dev_sms * per_sm;
    r->yield_every = yield_every;
    e = pkv::launch_resident(rp, p->kmap, p->vmap, r->grid, r->kstream);
    if (e != cudaSuccess) {
        resident_free(r);
        return cuda_fail(e);
    }
    r->launches = 1;
    r->running = true;
    s->resident = r;
    *out = r;
    return PKV_OK;
}

int pkv_resident_step(pkv_resident_t r, const void* q_h, const void* k_new_h, const void* v_new_h, float* out_h,
                      float* lse_h, int64_t wait_limit_ns) {
    NvtxRange range("pkv_resident_step");
    if (!r || !r->running || wait_limit_ns <= 0) return PKV_EINVAL;
    if (q_h) PKV_CUDA(cudaMemcpyAsync(r->q_d, q_h, r->q_bytes, cudaMemcpyHostToDevice, r->cstream));
    if (k_new_h) PKV_CUDA(cudaMemcpyAsync(r->k_new_d, k_new_h, r->new_bytes, cudaMemcpyHostToDevice, r->cstream));
    if (v_new_h) PKV_CUDA(cudaMemcpyAsync(r->v_new_d, v_new_h, r->new_bytes, cudaMemcpyHostToDevice, r->cstream));
    PKV_CUDA(cudaStreamSynchronize(r->cstream));
    if (r->yielded) {   // the kernel left the GPU after its last step: launch it again from this step
        pkv_plan_s* p = r->session->plan;
        r->rp.first_step = r->step + 1;
        host_store(&r->ctl_h->exited, 0u);
        PKV_CUDA(pkv::launch_resident(r->rp, p->kmap, p->vmap, r->grid, r->kstream));
        r->launch_first = r->step + 1;
        r->yielded = false;
        ++r->launches;
    }
    host_store(&r->ctl_h->requests, static_cast<uint32_t>(r->n_req));   // the requests staged for this step
    const uint32_t step = ++r->step;
    host_store(&r->ctl_h->step, step);
    const auto t0 = std::chrono::steady_clock::now();
    while (host_load(&r->ctl_h->done) < step) {
        // the kernel left its loop on an error (see pkv_status); a yield (3) comes only after this
        // step, whose outputs its last CTA is still publishing
        const uint32_t ex = host_load(&r->ctl_h->exited);
        if (ex != 0u && ex != 3u) return PKV_EDEVICE;
        if (std::chrono::steady_clock::now() - t0 > std::chrono::nanoseconds(wait_limit_ns)) return PKV_EDEVICE;
    }
    r->n_req = 0;   // applied by the step
    host_store(&r->ctl_h->requests, 0u);
    if (r->yield_every > 0 && (step - r->launch_first + 1) % static_cast<uint32_t>(r->yield_every) == 0) {
        // this launch's last step: the kernel is leaving; the GPU is free until the next step
        PKV_CUDA(cudaStreamSynchronize(r->kstream));
        if (host_load(&r->ctl_h->exited) != 3u) return PKV_EDEVICE;
        r->yielded = true;
    }
    if (out_h) PKV_CUDA(cudaMemcpyAsync(out_h, r->out_d, r->out_bytes, cudaMemcpyDeviceToHost, r->cstream));
    if (lse_h) PKV_CUDA(cudaMemcpyAsync(lse_h, r->lse_d, r->lse_bytes, cudaMemcpyDeviceToHost, r->cstream));
    if (out_h || lse_h) PKV_CUDA(cudaStreamSynchronize(r->cstream));
    return PKV_OK;
}

int pkv_resident_evict(pkv_resident_t r, const int32_t* rows_h, int32_t n) {
    if (!r || !r->running) return PKV_EINVAL;
    pkv_session_t s = r->session;
    int rc = check_slot_rows(s->active_h, s->plan->g.batch, rows_h, n, true);
    if (rc) return rc;
    if (r->n_req + n > PKV_RESIDENT_MAX_REQUESTS) return PKV_ENOSPACE;
    for (int32_t i = 0; i < n; ++i) {
        r->req_h[r->n_req++] = pkv::SlotRequest{rows_h[i], -1, 0, 0, nullptr, nullptr};
        s->active_h[rows_h[i]] = 0;
    }
    return PKV_OK;
}

int pkv_resident_admit(pkv_resident_t r, const int32_t* rows_h, const int32_t* lens_h, int32_t n, const void* k_src,
                       const void* v_src) {
    if (!r || !r->running) return PKV_EINVAL;
    pkv_session_t s = r->session;
    int rc = check_slot_rows(s->active_h, s->plan->g.batch, rows_h, n, false);
    if (rc) return rc;
    int64_t tokens = 0;
    if ((rc = check_admit_args(s->plan, lens_h, n, k_src, v_src, &tokens))) return rc;
    if (r->n_req + n > PKV_RESIDENT_MAX_REQUESTS) return PKV_ENOSPACE;
    int32_t src_tok = 0;
    for (int32_t i = 0; i < n; ++i) {
        r->req_h[r->n_req++] = pkv::SlotRequest{rows_h[i], lens_h[i], src_tok, -1, static_cast<const uint16_t*>(k_src),
                                                static_cast<const uint16_t*>(v_src)};
        src_tok += lens_h[i];
        s->active_h[rows_h[i]] = 1;
    }
    return PKV_OK;
}

int pkv_resident_stop(pkv_resident_t r) {
    if (!r) return PKV_EINVAL;
    if (!r->running) return PKV_OK;
    host_store(&r->ctl_h->stop, 1u);
    cudaError_t e = cudaStreamSynchronize(r->kstream);   // returns at once after a yield
    r->running = false;
    r->session->resident = nullptr;
    // the persistent route expects its queue counters rewound
    if (e == cudaSuccess) e = cudaMemset(r->session->plan->ctr, 0, 2 * sizeof(uint32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e);
    return host_load(&r->ctl_h->exited) == 2u ? PKV_EDEVICE : PKV_OK;
}

int pkv_resident_launches(pkv_resident_t r, int32_t* launches) {
    if (!r || !launches) return PKV_EINVAL;
    *launches = r->launches;
    return PKV_OK;
}

int pkv_resident_times(pkv_resident_t r, uint64_t* stamps_ns, int32_t capacity, int32_t* count) {
    if (!r || !count || r->running) return PKV_EINVAL;
    const int32_t n = static_cast<int32_t>(std::min<uint32_t>(r->step, static_cast<uint32_t>(r->times_cap)));
    *count = n;
    if (stamps_ns && capacity > 0 && n > 0)
        PKV_CUDA(cudaMemcpy(stamps_ns, r->times_d, sizeof(uint64_t) * 4 * std::min(n, capacity),
                            cudaMemcpyDeviceToHost));
    return PKV_OK;
}

void pkv_resident_destroy(pkv_resident_t r) {
    if (!r) return;
    if (r->running) pkv_resident_stop(r);
    resident_free(r);
}

void pkv_session_destroy(pkv_session_t s) {
    if (s && s->resident) {   // stop the kernel; the resident handle stays the caller's to destroy
        pkv_resident_s* r = s->resident;
        pkv_resident_stop(r);
        r->session = nullptr;
    }
    session_free(s);
}

}  // extern "C"

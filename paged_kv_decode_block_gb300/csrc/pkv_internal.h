// pkv_internal.h -- interface between the host library (planner, C ABI) and
// the CUDA kernels.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Record `e` as this thread's last CUDA error (what pkv_last_cuda_error
// returns) and return PKV_ECUDA.
int cuda_fail(cudaError_t e);

// Tokens per pipeline stage.  A page of page_size tokens is streamed as
// page_size / kBlockRows stages; page_size must be a multiple of it.
constexpr int kBlockRows = 16;

// Shared-memory scratch (floats) of one exact LSE merge: the planner keeps
// splits-per-(row, KV head) * G within it.
constexpr int kMergeCapFloats = 4096;

// Device-side bookkeeping of a plan (zeroed once at creation; kernels that
// change it put it back before they exit, so no host reset is needed between
// launches or graph replays).
struct DeviceCounters {
    uint32_t next_tile;  // persistent mode: next queue index to hand out
    uint32_t done_ctas;  // persistent mode: CTAs that found the queue empty
    uint32_t status;     // pkv_device_status_bits, sticky until pkv_status
    uint32_t pad;
};

enum Route : int32_t {
    kRouteDirect = 0,   // tile = (b, kvh) from blockIdx; whole row; finalise
    kRouteQueue = 1,    // tile = queue[blockIdx]
    kRoutePadded = 2,   // tile = (b, kvh, s) from blockIdx over B*Hkv*S_max
    kRoutePersistent = 3  // tiles from an atomic counter over the queue
};

// Per-CTA timeline of one attention launch (pkv_trace_enable): row blockIdx.x
// of kTraceWords words.  Times are %globaltimer ns (0: the phase did not occur).
// Every CTA writes its whole row, after the grid dependency wait, on every
// launch, so rows never mix two launches and need no reset between them.
enum TraceSlot : int {
    kTrTiles = 0,      // tiles this CTA ran
    kTrSm = 1,         // SM the CTA ran on
    kTrEntry = 2,      // kernel entry (before the grid dependency wait)
    kTrWaitDone = 3,   // grid dependency wait released
    kTrFirstBlock = 4, // consumer warp 0 holds its first block of the CTA's first tile
    kTrStreamEnd = 5,  // consumer warp 0 has reduced its last block of the last tile
    kTrCombineEnd = 6, // the last tile's four warp states are combined and written
    kTrArrived = 7,    // the last split tile's arrival counted (split routes)
    kTrMergeEnd = 8,   // this CTA merged a (row, KV head) as the last arrival: merge done
    kTrExit = 9,       // CTA done
    kTrLastTile = 10,  // (b << 40) | (kvh << 20) | split of the last tile
    kTraceWords = 12
};

struct AttnParams {
    const uint16_t* q;            // bf16 [B][Hq][D]
    const uint16_t* k_pages;      // bf16 [num_pages][page_size][Hkv][D]
    const uint16_t* v_pages;
    const int32_t* block_table;   // [B][max_pages]
    const int32_t* seq_lens;      // [B]
    const pkv_work_item* queue;   // [num_tiles] for queue / persistent routes
    const int32_t* row_start;     // [B] workspace slot of (b, kvh 0, split 0)
    const int32_t* row_splits;    // [B] slots per (b, kvh); 1 = tile finalises in place
    const int32_t* order;         // persistent route: queue index of the t-th tile handed out (or null)
    const int32_t* tiles_d;       // persistent route: tile count in device memory (overrides num_tiles)
    float* out;                   // [B][Hq][D]
    float* lse;                   // [B][Hq]
    float* ws_o;                  // [slots][G][D] normalised partial outputs
    float* ws_lse;                // [slots][G] partial LSE, log2 units
    uint32_t* arrive;             // [2][B*Hkv] fused-merge arrival, then departure counters
    DeviceCounters* ctr;
    int32_t B, Hq, Hkv, D, page_size, max_pages, num_pages;
    int32_t chunk_pages, max_splits, num_tiles;
    int32_t route;
    int32_t fused_merge;          // split tiles merge inside the attention launch
    int32_t all_merge;            // ... every split merges its share once all have arrived
                                  //     (cooperative one-wave launch); else the last arriver
    int32_t use_mma;              // block reduction on tensor cores (mma.sync) instead of FMA
    int32_t copy_lsu;             // stage K/V with cp.async from the producer warp instead of TMA
    int32_t queue_host_staged;    // queue / row_start / row_splits come from a host upload (never
                                  // written by a kernel), so they may be read before the grid
                                  // dependency wait
    int32_t no_empty_rows;        // queue / persistent routes: every row has tokens, so there is no
                                  // neutral state to write (0: look for empty rows after the tiles)
    float scale_log2;             // log2(e) / sqrt(D)
    uint64_t* trace;              // [grid][kTraceWords] per-CTA timeline, or null (off)
};

// Device planner of a continuous-decoding step (pkv_devplan.cu): page
// allocation from a device free list, then the plan for the lengths after the
// append, all on the GPU.
constexpr int kDevPlanMaxRows = 2048;
struct DevPlanParams {
    const int32_t* lens;        // [B] lengths before the append
    const int32_t* active;      // [B] 1: the row takes this step's token; 0: idle slot (null: all active)
    int32_t* table;             // [B][max_pages] device block table (entries filled in)
    const int32_t* free_list;   // [free_cap] free page ids, handed out in order
    uint32_t* free_state;       // {next index into free_list, pages still free}
    int32_t free_cap;
    pkv_work_item* queue;       // [queue_cap]
    int32_t* row_start;         // [B]
    int32_t* row_splits;        // [B]
    int32_t* order;             // [queue_cap] hand-out order, longest tile first
    int32_t* tiles;             // [1] tiles in this step's queue
    int32_t queue_cap;
    uint32_t* status;
    int32_t B, Hkv, page_size, max_pages, chunk;
};
cudaError_t launch_plan_step(const DevPlanParams& p, cudaStream_t stream);

// Attention launch: one of the four routes.  kmap / vmap are TMA descriptors
// of the K and V pools viewed as [page_size * num_pages][Hkv][D] (innermost D),
// box {64, 1, kBlockRows}, 128-byte swizzle.
cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             int grid, cudaStream_t stream, bool cooperative = false);
cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream);
// `active` (nullable, [B]): rows with 0 are idle slots and are left alone.
cudaError_t launch_append(const uint16_t* k_new, const uint16_t* v_new, uint16_t* k_pages,
                          uint16_t* v_pages, const int32_t* block_table, int32_t* seq_lens,
                          int B, int Hkv, int D, int page_size, int max_pages, int num_pages,
                          uint32_t* status, cudaStream_t stream, const int32_t* active = nullptr);
// One step of a host-planned continuous session in one launch: the new page
// of every row that starts one is entered in the table, the step's plan is
// copied from its pinned host staging into the plan's device buffer (the
// decode launched next reads it there), and the new token of every row is
// appended.  new_pages and plan_src are device views of mapped pinned host
// memory, read by the kernel over the host link; no copy engine is used.
struct AppendStepParams {
    const uint16_t* k_new;      // device bf16 [B][Hkv][D]
    const uint16_t* v_new;
    uint16_t* k_pages;
    uint16_t* v_pages;
    int32_t* block_table;       // [B][max_pages]
    int32_t* seq_lens;          // [B]
    const int32_t* new_pages;   // [B][2]: (table index, page id) of the row's new page, or index -1
    const int32_t* active;      // [B] 0: idle slot, left alone (null: all active)
    const int32_t* plan_src;    // plan staging (nullable: nothing to copy)
    int32_t* plan_dst;
    int64_t plan_words;         // int32 words of plan to copy
    uint32_t* status;
    int32_t B, Hkv, D, page_size, max_pages, num_pages;
};
cudaError_t launch_append_step(const AppendStepParams& p, cudaStream_t stream);
// Slot admit / evict (pkv_session_evict / pkv_session_admit / pkv_resident_*).
// One request per row; evictions are applied before admissions, each in the
// order listed.  32 bytes.
struct SlotRequest {
    int32_t row;
    int32_t len;                // -1: evict; >= 0: admit with a prompt of this many tokens
    int32_t src_tok;            // admit: the row's first token in k_src / v_src
    int32_t page_off;           // admit from the host pool: the row's first page in SlotParams::pages
    const uint16_t* k_src;      // admit: bf16 [tokens][Hkv][D] prompt K (device memory)
    const uint16_t* v_src;
};
struct SlotParams {
    const SlotRequest* req;     // [n] (device view; mapped pinned host memory)
    int32_t n;
    const int32_t* pages;       // host-pool admissions: the page ids chosen on the host (device view)
    int32_t* free_list;         // device free list ring [free_cap] (null: the host pool chose the pages)
    uint32_t* free_state;       // {index of its front, pages in it}
    int32_t free_cap;
    int32_t* table;             // [B][max_pages]
    int32_t* lens;              // [B]
    int32_t* active;            // [B]
    uint16_t* k_pages;
    uint16_t* v_pages;
    uint32_t* status;
    int32_t B, Hkv, D, page_size, max_pages, num_pages;
};
// The bookkeeping (one CTA), then the copy of the admitted prompts (a grid).
cudaError_t launch_slot_requests(const SlotParams& p, cudaStream_t stream);

// Bounded-wait self-test (see pkv_selftest_wait): result[3] = {wait returned true,
// abort flag raised, second wait returned true}.
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, int* result, cudaStream_t stream);

// Resident continuous decoding (pkv_resident_*): one cooperative launch that
// stays on the GPU and runs a step (plan, append, decode) each time the host
// publishes one.  The control block lives in mapped pinned host memory.
struct ResidentCtl {
    uint32_t step;       // host: the last step it has published (1, 2, ...)
    uint32_t stop;       // host: 1 = leave the loop instead of waiting for another step
    uint32_t done;       // kernel: the last step whose outputs are written
    uint32_t exited;     // kernel: 1 once it has left the loop; 2 if it left on an error; 3 if it
                         // yielded the GPU after yield_every steps (the host relaunches it)
    uint32_t requests;   // host: slot requests to apply at the start of the published step
    uint32_t pad[3];
};
// grid_sync words (device memory, zero before the launch)
enum ResidentSync {
    kSyncCount = 0, kSyncGen = 1,   // grid barrier: arrivals, generation
    kSyncCmd = 2,                   // the step's command (go / stop / fail), set by CTA 0
    kSyncAbort = 3,                 // a bounded wait ran out somewhere: every CTA leaves
    kSyncReq = 4,                   // slot requests of the step
    kSyncDone = 5,                  // CTAs done with the step's decode (the last one publishes)
    kSyncWords = 6
};
struct ResidentParams {
    AttnParams attn;            // persistent route over the device plan below
    DevPlanParams plan;         // allocation + plan of each step (lengths before its append)
    SlotParams slots;           // the step's slot requests (req, n from the control block)
    const uint16_t* k_new;      // device bf16 [B][Hkv][D]: the step's new token per row
    const uint16_t* v_new;
    uint16_t* k_pages_w;        // the pools and lengths, writable (the append)
    uint16_t* v_pages_w;
    int32_t* lens_w;
    ResidentCtl* ctl;           // device view of the mapped control block
    uint32_t* grid_sync;        // [kSyncWords]
    uint64_t* times;            // [times_cap][4] globaltimer of a step: seen, planned, appended, published
    int32_t times_cap;
    uint64_t idle_limit_ns;     // longest wait for the host's next step
    uint32_t* row_ready;        // [B] the last step whose append of the row has landed
    uint32_t first_step;        // the first step this launch runs
    int32_t yield_every;        // leave the GPU after this many steps of the launch (0: never)
};
cudaError_t launch_resident(const ResidentParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                            cudaStream_t stream);
int resident_ctas_per_sm(int D, int G, bool mma);
// Resident CTAs per SM of the attention kernel for this (D, G); 0 if unsupported.
int attention_ctas_per_sm(int D, int G, bool mma);
bool shape_supported(int D, int G);

}  // namespace pkv

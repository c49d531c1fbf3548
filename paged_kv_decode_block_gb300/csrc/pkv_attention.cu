// pkv_attention.cu -- paged GQA decode attention kernels for GB300 (sm_103a).
//
// Method: "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM
// Serving on Commodity GPUs" (gist.science summary), Technical Summary,
// Methodology section 1 "Native Block-Table Decode Engine":
//   * one pass over a KV head serves its whole group of G = Hq/Hkv query heads;
//   * K and V are read in place through the block table ("Layout");
//   * a split computes the partial online-softmax state of a disjoint page
//     range and a merge combines the states exactly ("Sequence Splitting");
//   * split ranges follow the row's true length; an empty split writes the
//     neutral state and reads no KV ("Row-Local Bounds");
//   * tiles come from a compact queue of non-empty (row, KV head, split)
//     intervals ("Compact Workqueue").
// The persistent route drains that queue with an atomic counter, like the
// worker of "GPUOS" (arXiv 2604.17861, section 4.1 "Persistent Kernel
// Executor"), with the grid sized to the SM count as in "WPK persistent kernel"
// (dotwave.ai, "What a persistent kernel is").
//
// GB300 design.  The kernel streams every KV byte once from HBM:
//   * one CTA per tile: 4 consumer warps + 4 producer warps;
//   * the producers resolve the block table (32 entries per coalesced load,
//     prefetched one batch ahead) and stream 16-token blocks of K and V into
//     a ring of 10-16 shared-memory stages (about 80-96 KB per CTA, two CTAs
//     per SM), in a 128-byte-swizzled layout with L2 evict-first: 16-byte
//     cp.async from all producer lanes (default) or TMA boxes
//     (cp.async.bulk.tensor); completion tracked by mbarriers;
//   * the launch may overlap the previous kernel's tail (programmatic
//     dependent launch): nothing is read before the grid dependency wait
//     except the host-staged queue entry, and the tile's first blocks are
//     warmed in L2 there;
//   * each consumer warp owns every 4th block and keeps a private
//     online-softmax state (running max, sum, fp32 accumulator), so the loop has
//     no CTA-wide barrier; the four states are merged with the exact LSE rule at
//     the end of the tile, and a split tile's partial goes to the workspace
//     where the last-arriving split of its (row, KV head) merges them all (or,
//     in a cooperative launch, every split merges a share);
//   * two interchangeable block reductions (template MMA):
//       - FMA: CUDA cores; D/8 lanes cover a K row in 16-byte slices and the G
//         dot products are summed by a transposing butterfly;
//       - MMA: warp-level mma.sync m16n8k16 bf16 with fp32 accumulation for
//         S^T = K Q^T (16 tokens x the query group, padded to 8 columns) and for
//         O^T += V^T P^T.  P (in [0,1]) is split into bf16 hi + lo parts that
//         ride in the padding columns (or a second column tile when G = 8), so
//         P V keeps about 16 mantissa bits; K and V come from shared memory with
//         ldmatrix (conflict-free under the swizzle) straight into registers,
//         and the stage is released before any arithmetic, so stages are held
//         only briefly and the ring stays full of loads in flight.  This also
//         cuts the issued instructions per block about six-fold against FMA;
//   * scores stay in the log2 domain (scale log2(e)/sqrt(D) applied in fp32);
//     exp2f is CUDA's own function; all accumulation is fp32.
// Every wait on an mbarrier is bounded (kWaitLimitNs): on expiry the kernel
// sets PKV_DEV_TIMEOUT, poisons the tile, stops waiting and drains its own
// copies before exit.  Bad page ids set PKV_DEV_PAGE_OOB and poison the tile;
// no access is made through them.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pkv_devplan.cuh"
#include "pkv_internal.h"
#include "pkv_slots.cuh"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
// Block j is staged by producer warp j % kProducerWarps.  One producer warp
// keeps only a few blocks' copies in flight, and that caps a CTA's stream
// rate well below its share of HBM: a CTA alone on an SM streamed 35 %
// faster with four producer warps than with two, and the MMA consumers still
// fit the 128 registers a thread that two 256-thread CTAs per SM leave.
constexpr int kProducerWarps = 4;
constexpr int kThreads = (kConsumerWarps + kProducerWarps) * 32;
constexpr int kPrefetchBlocks = 8;   // blocks of a tile warmed in L2 before the grid dependency wait
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr unsigned kFull = 0xffffffffu;
constexpr float kLn2 = 0.69314718055994530942f;

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, for at most
// kWaitLimitNs.  On expiry: flag the status word, raise the CTA's abort flag
// (later waits of the CTA then return at once) and return false.
__device__ __noinline__ bool mbar_wait_slow(uint64_t* bar, uint32_t parity, uint32_t* status,
                                            volatile int* abort, uint64_t limit_ns = kWaitLimitNs) {
    if (abort && *abort) return false;
    const uint64_t start = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - start > limit_ns) {
            atomicOr(status, static_cast<uint32_t>(PKV_DEV_TIMEOUT));
            if (abort) *abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t* status, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, status, abort);
}

// Bounded wait (one thread) until the counter at `ctr` reaches `target`, read
// with acquire semantics at GPU scope.  On expiry: flag the status word, raise
// the CTA's abort flag and return false.
__device__ __noinline__ bool wait_count(const uint32_t* ctr, uint32_t target, uint32_t* status, volatile int* abort) {
    if (abort && *abort) return false;
    const uint64_t start = globaltimer_ns();
    while (true) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
        if (v >= target) return true;
        if (globaltimer_ns() - start > kWaitLimitNs) {
            atomicOr(status, static_cast<uint32_t>(PKV_DEV_TIMEOUT));
            if (abort) *abort = 1;
            return false;
        }
        __nanosleep(32);
    }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t policy;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
    return policy;
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// 16-byte asynchronous global -> shared copy through L2 only, with an L2 policy.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
                 : "memory");
}

// 16-byte asynchronous global -> shared copy through L2 only (generic proxy:
// no proxy fence is needed against plain stores of other CTAs).
__device__ __forceinline__ void cp_async16_plain(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

// Programmatic dependent launch: wait until the grids this launch depends on
// have completed and their memory is visible (a no-op for an ordinary launch),
// and let the next grid in the stream start launching its CTAs.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Hint: bring the 128-byte line holding `p` into L2 (no data returns; a stale
// or unused prefetch changes nothing but the cache).
__device__ __forceinline__ void prefetch_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

__device__ __forceinline__ int32_t ld_volatile_i32(const int32_t* p) {
    int32_t v;
    asm volatile("ld.volatile.global.s32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release_sys(uint32_t* p, uint32_t v) {
    asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_sc_sys() { asm volatile("fence.sc.sys;" ::: "memory"); }

// Order earlier generic-proxy accesses (as acquired from another CTA) before
// later async-proxy (TMA) accesses to global memory.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Release / acquire fence at GPU scope (message passing between CTAs).
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Atomic add with acquire semantics at GPU scope; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acquire_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acquire.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Arrive on `bar` once every cp.async this thread has issued so far has landed
// (the arrival counts against the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1])
                 : "r"(addr)
                 : "memory");
}

// D (16x8 fp32) += A (16x16 bf16, row-major) * B (16x8 bf16, column-major)
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 8 packed bf16 (one 16-byte vector) -> 8 floats.  bf16 is the top half of an
// IEEE binary32, so widening is a shift or a mask.
__device__ __forceinline__ void unpack_bf16x8(const uint4& raw, float (&f)[8]) {
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

// Byte offset, inside one K or V stage, of the 16-byte chunk holding token
// row's elements [d, d + 8) (d a multiple of 8).  A stage holds D/64 halves of
// [16 rows][128 B]; TMA's 128-byte swizzle stores chunk c of row r at chunk
// c ^ (r % 8), so 8 rows read at one chunk index hit 8 distinct bank groups.
__device__ __forceinline__ uint32_t swz(int row, int d) {
    return static_cast<uint32_t>((d >> 6) * (kBlockRows * 128) + row * 128 + ((((d & 63) >> 3) ^ (row & 7)) << 4));
}

// Transposing butterfly over the lanes of one row group.  Starting from N
// per-lane partial sums (one per head), each exchange with partner lane^MASK
// trades half of the values, so after log2(N) steps a lane holds one head's
// sum; the remaining steps are plain butterflies.  Returns the full sum of
// head (lane % L) / (L / N) where L = 2 * first MASK.
template <int MASK, int N>
struct Butterfly {
    static __device__ __forceinline__ float run(float* v, int lane) {
        if constexpr (MASK == 0) {
            static_assert(N == 1, "group wider than the row's lanes");
            return v[0];
        } else if constexpr (N > 1) {
            const bool upper = (lane & MASK) != 0;
#pragma unroll
            for (int i = 0; i < N / 2; ++i) {
                const float send = upper ? v[i] : v[i + N / 2];
                const float keep = upper ? v[i + N / 2] : v[i];
                v[i] = keep + __shfl_xor_sync(kFull, send, MASK);
            }
            return Butterfly<MASK / 2, N / 2>::run(v, lane);
        } else {
            v[0] += __shfl_xor_sync(kFull, v[0], MASK);
            return Butterfly<MASK / 2, 1>::run(v, lane);
        }
    }
};

// ------------------------------------------------------------------ layout

template <int D, int G>
struct Cfg {
    // FMA form
    static constexpr int L = D / 8;                 // lanes per K/V row (16 B each)
    static constexpr int R = 32 / L;                // rows per warp step
    static constexpr int kSteps = kBlockRows / R;   // warp steps per 16-row block
    static constexpr int HG = L / G;                // lanes holding the same head
    // both forms
    static constexpr int kMatBytes = kBlockRows * D * 2;            // one K or V stage
    static constexpr uint32_t kStageBytes = 2u * kMatBytes;         // K + V
    // MMA form: P^T column tiles (hi and lo parts share one tile while 2G <= 8)
    static constexpr int NPV = (2 * G <= 8) ? 1 : 2;
    // Ring depth: about 80-96 KB of K/V in flight per CTA, two CTAs per SM.
    static constexpr int kStages = D == 128 ? (G == 8 ? 10 : 12) : 16;
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G >= 1 && G <= 8 && G <= L, "group size");
};

template <int D, int G>
struct Smem {
    static constexpr int kStages = Cfg<D, G>::kStages;
    alignas(1024) uint8_t k[kStages][Cfg<D, G>::kMatBytes];
    alignas(1024) uint8_t v[kStages][Cfg<D, G>::kMatBytes];
    alignas(16) uint16_t pt[kConsumerWarps][Cfg<D, G>::NPV * 2 * 8 * 8];   // P^T tiles, bf16 (MMA form)
    float p[kConsumerWarps][kBlockRows * G];   // softmax weights of the block (FMA form)
    alignas(16) float acc[kConsumerWarps][G * D];   // per-warp states for the end-of-tile merge
    float m[kConsumerWarps][G];
    float l[kConsumerWarps][G];
    float merge_m[G], merge_inv[G];
    int merge_nan_h[G];         // per head: a split's LSE was NaN (written once per merge, no reset)
    int poisoned[kConsumerWarps];
    int bad[kStages];
    uint32_t issued[kStages];   // 1 + use index of the last TMA issued into each stage
    int abort;                  // a wait of this CTA ran out: stop waiting, drain, finish
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int tile_slot[2];
    int tile_fin, tile_splits;  // the finished tile's finalize flag and split count
    int tile_base;              // workspace slot of split 0 of the finished tile's (row, KV head)
    int sync_ok;                // resident kernel: the last grid barrier / host wait succeeded
    int append_page, append_pos;
    uint64_t tr[kTraceWords];   // this launch's timeline row (when p.trace is set), flushed at exit
};

template <int D, int G>
constexpr size_t smem_bytes() {
    return sizeof(Smem<D, G>) + 1024;   // + room to align the base to 1024 B
}

__device__ __forceinline__ uint32_t smid() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

// Timeline stamp of thread 0 into the CTA's row (pkv_trace_enable); a uniform
// branch on a kernel parameter when tracing is off.
template <int D, int G>
__device__ __forceinline__ void trace_stamp(Smem<D, G>& sm, const AttnParams& p, int slot) {
    if (p.trace && threadIdx.x == 0) sm.tr[slot] = globaltimer_ns();
}

struct TileWork {
    int b, kvh;
    int t0, t1;        // token range [t0, t1) of row b (clipped to N_b)
    int t_stream;      // tokens [t0, t_stream) are streamed (whole planned pages for queue tiles)
    int split, page_begin, page_end;
    int slot;          // workspace slot (split tiles)
    int finalize;      // 1: write out/lse directly
    int splits;        // splits of (b, kvh)
    int poisoned;      // plan and device lengths disagree
    int lazy;          // t1 / slot / finalize / splits / poisoned still to be read (tile_finish)
};

__device__ __forceinline__ int stream_blocks(const TileWork& tw) {
    const int n = tw.t_stream > tw.t0 ? tw.t_stream - tw.t0 : 0;
    return (n + kBlockRows - 1) / kBlockRows;
}

// ------------------------------------------------------------------ FMA block reduction

template <int D, int G>
struct FmaState {
    float qf[G][8];    // this lane's 8-element slice of every query head, pre-scaled
    float m[G], l[G];  // running max / sum (log2 domain), warp-uniform
    float m_mine;      // running max of the head this lane reduces
    float acc[G][8];   // this lane's slice of the unnormalised output
};

template <int D, int G>
__device__ __forceinline__ void fma_init(FmaState<D, G>& st, const AttnParams& p, const TileWork& tw, int lane) {
    using C = Cfg<D, G>;
    const int sub = lane % C::L;
    const uint16_t* qrow = p.q + (static_cast<size_t>(tw.b) * p.Hq + tw.kvh * G) * D + sub * 8;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow + g * D));
        unpack_bf16x8(raw, st.qf[g]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            st.qf[g][e] *= p.scale_log2;
            st.acc[g][e] = 0.f;
        }
        st.m[g] = -INFINITY;
        st.l[g] = 0.f;
    }
    st.m_mine = -INFINITY;
}

template <int D, int G>
__device__ __forceinline__ void fma_block(FmaState<D, G>& st, const uint8_t* ks, const uint8_t* vs,
                                          float* __restrict__ ps, int valid, int lane) {
    using C = Cfg<D, G>;
    const int sub = lane % C::L;
    const int rg = lane / C::L;
    const int my_g = sub / C::HG;

    float sc[C::kSteps];
#pragma unroll
    for (int s = 0; s < C::kSteps; ++s) {
        const int row = s * C::R + rg;
        const uint4 raw = *reinterpret_cast<const uint4*>(ks + swz(row, sub * 8));
        float kf[8];
        unpack_bf16x8(raw, kf);
        float dot[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float a = st.qf[g][0] * kf[0];
#pragma unroll
            for (int e = 1; e < 8; ++e) a = fmaf(st.qf[g][e], kf[e], a);
            dot[g] = a;
        }
        const float sv = Butterfly<C::L / 2, G>::run(dot, lane);
        sc[s] = row < valid ? sv : -INFINITY;
    }

    float bm = sc[0];
#pragma unroll
    for (int s = 1; s < C::kSteps; ++s) bm = fmaxf(bm, sc[s]);
#pragma unroll
    for (int mask = C::L; mask < 32; mask <<= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, mask));
    float alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float bmg = __shfl_sync(kFull, bm, g * C::HG);
        const float mn = fmaxf(st.m[g], bmg);
        alpha[g] = exp2f(st.m[g] - mn);   // m = -inf on the first block: alpha = 0
        st.m[g] = mn;
    }
    st.m_mine = fmaxf(st.m_mine, bm);

    float pr[C::kSteps];
    float psum = 0.f;
#pragma unroll
    for (int s = 0; s < C::kSteps; ++s) {
        pr[s] = exp2f(sc[s] - st.m_mine);   // masked rows: exp2(-inf) = 0
        psum += pr[s];
    }
#pragma unroll
    for (int mask = C::L; mask < 32; mask <<= 1) psum += __shfl_xor_sync(kFull, psum, mask);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        st.l[g] = st.l[g] * alpha[g] + __shfl_sync(kFull, psum, g * C::HG);
#pragma unroll
        for (int e = 0; e < 8; ++e) st.acc[g][e] *= alpha[g];
    }

    if (sub % C::HG == 0) {
#pragma unroll
        for (int s = 0; s < C::kSteps; ++s) ps[(s * C::R + rg) * G + my_g] = pr[s];
    }
    __syncwarp();
#pragma unroll
    for (int s = 0; s < C::kSteps; ++s) {
        const int row = s * C::R + rg;
        if (row < valid) {   // rows past N_b may hold stale, even non-finite, data
            const uint4 raw = *reinterpret_cast<const uint4*>(vs + swz(row, sub * 8));
            float vf[8];
            unpack_bf16x8(raw, vf);
            float pv[G];
#pragma unroll
            for (int g = 0; g < G; ++g) pv[g] = ps[row * G + g];
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) st.acc[g][e] = fmaf(pv[g], vf[e], st.acc[g][e]);
        }
    }
    __syncwarp();
}

// Publish the warp's state (m, l, unnormalised output) for the end-of-tile merge.
template <int D, int G>
__device__ __forceinline__ void fma_publish(FmaState<D, G>& st, Smem<D, G>& sm, int warp, int lane) {
    using C = Cfg<D, G>;
    const int sub = lane % C::L;
#pragma unroll
    for (int mask = C::L; mask < 32; mask <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) st.acc[g][e] += __shfl_xor_sync(kFull, st.acc[g][e], mask);
    if (lane < C::L) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) sm.acc[warp][g * D + sub * 8 + e] = st.acc[g][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            sm.m[warp][g] = st.m[g];
            sm.l[warp][g] = st.l[g];
        }
    }
}

// ------------------------------------------------------------------ MMA block reduction
//
// Fragment layout of mma.m16n8k16 (gid = lane / 4, tig = lane % 4):
//   A rows gid, gid+8 / cols 2tig(+1), 2tig+8(+1);  B rows (k) 2tig(+1), 2tig+8(+1) / col gid;
//   C rows gid, gid+8 / cols 2tig, 2tig+1.
// QK: S^T[token][column] with column n = query head n (n < G, the rest zero).
// PV: O^T[d][column]: column n < G is head n's hi part; the lo parts sit in
// columns G..2G-1 (2G <= 8) or in a second column tile (G = 8).

template <int D, int G>
struct MmaState {
    uint32_t qb[D / 16][2];                  // B fragments of Q^T
    float m[2];                              // running max of heads 2tig, 2tig+1 (log2 domain)
    float l[2];                              // this lane's share of their running sums
    float o[Cfg<D, G>::NPV][D / 16][4];      // O^T accumulators
};

template <int D, int G>
__device__ __forceinline__ void mma_init(MmaState<D, G>& st, const AttnParams& p, const TileWork& tw, int lane) {
    const int gid = lane >> 2, tig = lane & 3;
    const uint16_t* qh = p.q + (static_cast<size_t>(tw.b) * p.Hq + tw.kvh * G + (gid < G ? gid : 0)) * D;
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt) {
        st.qb[kt][0] = gid < G ? __ldg(reinterpret_cast<const uint32_t*>(qh + kt * 16 + 2 * tig)) : 0u;
        st.qb[kt][1] = gid < G ? __ldg(reinterpret_cast<const uint32_t*>(qh + kt * 16 + 8 + 2 * tig)) : 0u;
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        st.m[c] = -INFINITY;
        st.l[c] = 0.f;
    }
#pragma unroll
    for (int t = 0; t < Cfg<D, G>::NPV; ++t)
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) st.o[t][mt][i] = 0.f;
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ float bf16_value(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

template <int D, int G>
__device__ __forceinline__ void mma_block(MmaState<D, G>& st, uint8_t* ks, uint8_t* vs, uint64_t* empty,
                                          uint16_t* pt, int valid, int lane, float scale_log2) {
    using C = Cfg<D, G>;
    const int gid = lane >> 2, tig = lane & 3;
    const int j = lane >> 3, r8 = lane & 7;
    const uint32_t ka = smem_addr(ks), va = smem_addr(vs);

    // Rows past N_b may hold stale, even non-finite, data (0 * inf = NaN in P V):
    // zero them in the stage first.
    if (valid < kBlockRows) {
        for (int idx = lane; idx < (kBlockRows - valid) * (D / 8); idx += 32) {
            const int row = valid + idx / (D / 8);
            *reinterpret_cast<uint4*>(vs + swz(row, (idx % (D / 8)) * 8)) = make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_shared();   // the next TMA into this stage is ordered after these writes
        __syncwarp();
    }
    // The whole block moves to registers as mma fragments, and the stage goes
    // straight back to the producer: a stage is held for a few dozen cycles,
    // not for the block's arithmetic, so the ring stays full of loads in flight.
    uint32_t kf[D / 16][4], vf[D / 16][4];
    {
        const int row = r8 + 8 * (j & 1);
        const int tok = r8 + 8 * (j >> 1);
#pragma unroll
        for (int kt = 0; kt < D / 16; ++kt) ldsm_x4(kf[kt], ka + swz(row, kt * 16 + 8 * (j >> 1)));
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) ldsm_x4_trans(vf[mt], va + swz(tok, mt * 16 + 8 * (j & 1)));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty);

    // S^T = K Q^T over D in steps of 16
    float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kt = 0; kt < D / 16; ++kt) mma_16816(s, kf[kt], st.qb[kt][0], st.qb[kt][1]);
    const bool r0 = gid < valid, r1 = gid + 8 < valid;
    s[0] = r0 ? s[0] * scale_log2 : -INFINITY;
    s[1] = r0 ? s[1] * scale_log2 : -INFINITY;
    s[2] = r1 ? s[2] * scale_log2 : -INFINITY;
    s[3] = r1 ? s[3] * scale_log2 : -INFINITY;

    // online softmax for the lane's two columns
    float bm0 = fmaxf(s[0], s[2]), bm1 = fmaxf(s[1], s[3]);
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
        bm0 = fmaxf(bm0, __shfl_xor_sync(kFull, bm0, x));
        bm1 = fmaxf(bm1, __shfl_xor_sync(kFull, bm1, x));
    }
    const float mn0 = fmaxf(st.m[0], bm0), mn1 = fmaxf(st.m[1], bm1);
    const float al0 = exp2f(st.m[0] - mn0), al1 = exp2f(st.m[1] - mn1);   // first block: 0
    st.m[0] = mn0;
    st.m[1] = mn1;
    const float p0 = exp2f(s[0] - mn0), p1 = exp2f(s[1] - mn1);   // token gid
    const float p2 = exp2f(s[2] - mn0), p3 = exp2f(s[3] - mn1);   // token gid + 8
    st.l[0] = st.l[0] * al0 + (p0 + p2);
    st.l[1] = st.l[1] * al1 + (p1 + p3);

    // P^T into shared memory as bf16 hi/lo parts: pt[tile][half][column][8 tokens]
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        const int h = 2 * tig + c;
        if (h < G) {
            const float pa = c ? p1 : p0, pb = c ? p3 : p2;
            const uint16_t ha = bf16_bits(pa), hb = bf16_bits(pb);
            const uint16_t la = bf16_bits(pa - bf16_value(ha)), lb = bf16_bits(pb - bf16_value(hb));
            constexpr int lt = C::NPV == 1 ? 0 : 1;
            const int ln = C::NPV == 1 ? G + h : h;
            pt[((0 * 2 + 0) * 8 + h) * 8 + gid] = ha;
            pt[((0 * 2 + 1) * 8 + h) * 8 + gid] = hb;
            pt[((lt * 2 + 0) * 8 + ln) * 8 + gid] = la;
            pt[((lt * 2 + 1) * 8 + ln) * 8 + gid] = lb;
        }
    }

    // rescale O^T by the alpha of the head each of the lane's columns belongs to
    float a0, a1;
    if constexpr (G == 1) {
        a0 = a1 = __shfl_sync(kFull, al0, lane & ~3);
    } else if constexpr (C::NPV == 1) {
        const int h0 = (2 * tig) & (G - 1);
        const int src = (lane & ~3) | (h0 >> 1);
        a0 = __shfl_sync(kFull, al0, src);
        a1 = __shfl_sync(kFull, al1, src);
    } else {
        a0 = al0;
        a1 = al1;
    }
#pragma unroll
    for (int t = 0; t < C::NPV; ++t)
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
            st.o[t][mt][0] *= a0;
            st.o[t][mt][1] *= a1;
            st.o[t][mt][2] *= a0;
            st.o[t][mt][3] *= a1;
        }

    __syncwarp();

    uint32_t pb[C::NPV][2];
#pragma unroll
    for (int t = 0; t < C::NPV; ++t)
        ldsm_x2(pb[t], smem_addr(pt) + (((t * 2 + ((lane >> 3) & 1)) * 8 + (lane & 7)) * 16));

    // O^T += V^T P^T over D in tiles of 16
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int t = 0; t < C::NPV; ++t) mma_16816(st.o[t][mt], vf[mt], pb[t][0], pb[t][1]);
    __syncwarp();   // pt is rewritten by the next block
}

template <int D, int G>
__device__ __forceinline__ void mma_publish(MmaState<D, G>& st, Smem<D, G>& sm, int warp, int lane) {
    using C = Cfg<D, G>;
    const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) st.l[c] += __shfl_xor_sync(kFull, st.l[c], x);
    // fold the lo parts into the hi parts
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
        float f[4];
        if constexpr (G == 1) {
            f[0] = st.o[0][mt][0] + st.o[0][mt][1];
            f[2] = st.o[0][mt][2] + st.o[0][mt][3];
            f[1] = f[3] = 0.f;
        } else if constexpr (C::NPV == 1) {
            const int src = (lane & ~3) | ((tig + G / 2) & 3);
#pragma unroll
            for (int i = 0; i < 4; ++i) f[i] = st.o[0][mt][i] + __shfl_sync(kFull, st.o[0][mt][i], src);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) f[i] = st.o[0][mt][i] + st.o[1][mt][i];
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int h = 2 * tig + c;
            if (h < G) {
                sm.acc[warp][h * D + mt * 16 + gid] = f[c];
                sm.acc[warp][h * D + mt * 16 + gid + 8] = f[2 + c];
            }
        }
    }
    if (gid == 0) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int h = 2 * tig + c;
            if (h < G) {
                sm.m[warp][h] = st.m[c];
                sm.l[warp][h] = st.l[c];
            }
        }
    }
}

// ------------------------------------------------------------------ merges

// Write the neutral state (out = 0, lse = -inf) for every query head of row b.
__device__ void write_neutral_row(const AttnParams& p, int b, int tid, int nthreads) {
    for (int i = tid; i < p.Hq * p.D; i += nthreads) p.out[static_cast<size_t>(b) * p.Hq * p.D + i] = 0.f;
    for (int i = tid; i < p.Hq; i += nthreads) p.lse[static_cast<size_t>(b) * p.Hq + i] = -INFINITY;
}

// Exact LSE merge of the `ns` partial states of (b, kvh) into out / lse
// (M = max_s lse_s, w_s = 2^(lse_s - M) / sum_s 2^(lse_s - M), out = sum_s w_s o_s).
// Must be called by every thread of the CTA.  Partials come from other CTAs,
// so they are read through L2 (ld.cg).  `wsm` is shared scratch of
// kMergeCapFloats floats (the planner keeps ns * G within it).
template <int D, int G>
__device__ void merge_unit(const AttnParams& p, int b, int kvh, int ns, float* wsm, float* m_s, float* inv_s,
                           int* nan_s) {
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const size_t base = static_cast<size_t>(p.row_start[b]) + static_cast<size_t>(kvh) * ns;
    if (tid == 0) *nan_s = 0;
    __syncthreads();
    for (int i = tid; i < ns * G; i += nthreads) {
        const float ls = __ldcg(p.ws_lse + base * G + i);
        if (isnan(ls)) *nan_s = 1;
        wsm[i] = ls;
    }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int s = 0; s < ns; ++s) M = fmaxf(M, wsm[s * G + tid]);
        float wsum = 0.f;
        if (M != -INFINITY)
            for (int s = 0; s < ns; ++s) wsum += exp2f(wsm[s * G + tid] - M);
        m_s[tid] = M;
        inv_s[tid] = M != -INFINITY ? 1.f / wsum : 0.f;
        const float lse2 = M != -INFINITY ? M + log2f(wsum) : -INFINITY;
        p.lse[static_cast<size_t>(b) * p.Hq + kvh * G + tid] = *nan_s ? NAN : lse2 * kLn2;
    }
    __syncthreads();
    for (int i = tid; i < ns * G; i += nthreads) {
        const int g = i % G;
        wsm[i] = m_s[g] != -INFINITY ? exp2f(wsm[i] - m_s[g]) * inv_s[g] : 0.f;
    }
    __syncthreads();
    const bool nan = *nan_s != 0;
    for (int i = tid; i < G * D / 4; i += nthreads) {
        const int g = i / (D / 4), d = (i % (D / 4)) * 4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float* src = p.ws_o + (base * G + g) * D + d;
#pragma unroll 8
        for (int s = 0; s < ns; ++s) {
            const float w = wsm[s * G + g];
            const float4 o = __ldcg(reinterpret_cast<const float4*>(src + static_cast<size_t>(s) * G * D));
            acc.x = fmaf(w, o.x, acc.x);
            acc.y = fmaf(w, o.y, acc.y);
            acc.z = fmaf(w, o.z, acc.z);
            acc.w = fmaf(w, o.w, acc.w);
        }
        if (nan) acc = make_float4(NAN, NAN, NAN, NAN);
        *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(b) * p.Hq + kvh * G + g) * D + d) = acc;
    }
    __syncthreads();
}

// Merge staging geometry: the weights, then the partials, in the idle stage
// buffers; ns <= kMaxSplits take the one-pass path.
template <int D, int G>
struct MergeCfg {
    static constexpr int kSplitBytes = G * D * 4;
    static constexpr int kWeightBytes = 2048;   // [64][G] floats at most
    static constexpr int kScratch = Cfg<D, G>::kStages * Cfg<D, G>::kMatBytes * 2;
    static constexpr int kCap = (kScratch - kWeightBytes) / kSplitBytes;
    static constexpr int kMaxSplits = kCap < 64 ? kCap : 64;
    static_assert(64 * G * 4 <= kWeightBytes, "merge staging");
};

// The fused merge of the last-arriving CTA for up to MergeCfg::kMaxSplits
// splits.  The ns partial outputs of (b, kvh) are contiguous in the
// workspace; every thread copies its 16-byte pieces of them into the CTA's
// idle stage buffers with cp.async (the fastest way into one SM: per-thread
// loads are held back by the outstanding-request limit, and the bulk-copy
// engine measured slower).  The LSEs come in meanwhile, one warp per head
// holding splits lane and lane + 32; the max, sum and weights are shuffles.
// The weighted sum runs once everything has landed: T = kThreads / (G*D/4)
// lane groups share one float4 of the output (group `part` taking splits
// part, part + T, ...; a quarter warp reads 128 contiguous bytes), so all
// threads add, and the T part sums are added with a fixed butterfly: the
// result is the same on every launch.  Same arithmetic as merge_unit up to
// the order of the additions; all CTA threads call it.
template <int D, int G>
__device__ void merge_unit_onepass(Smem<D, G>& sm, const AttnParams& p, int b, int kvh, int ns, int base_slot) {
    using MC = MergeCfg<D, G>;
    constexpr int kOut = G * D / 4;       // float4 outputs of (b, kvh)
    constexpr int T = kThreads / kOut;    // lane groups per output
    constexpr int W = 32 / T;             // outputs per warp
    static_assert(kThreads % kOut == 0 && T >= 1 && T <= 32 && (T & (T - 1)) == 0, "merge lane split");
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int out = warp * W + lane % W, part = lane / W;
    const int g_out = out / (D / 4), d = (out % (D / 4)) * 4;
    const size_t base = static_cast<size_t>(base_slot);
    float* w = reinterpret_cast<float*>(&sm.k[0][0]);   // [ns][G] weights
    float* obuf = reinterpret_cast<float*>(&sm.k[0][0] + MC::kWeightBytes);   // [ns][G][D] partials

    const float ls_first = warp < G && lane < ns ? __ldcg(p.ws_lse + (base + lane) * G + warp) : -INFINITY;
    const float ls_first_hi = warp < G && lane + 32 < ns ? __ldcg(p.ws_lse + (base + lane + 32) * G + warp) : -INFINITY;
    {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.ws_o + base * G * D);
        const uint32_t dst = smem_addr(obuf);
        const int vecs = ns * (MC::kSplitBytes / 16);
        for (int i = tid; i < vecs; i += kThreads) cp_async16_plain(dst + i * 16, src + static_cast<size_t>(i) * 16);
    }
    for (int g = warp; g < G; g += kThreads / 32) {
        const float ls = g == warp ? ls_first : lane < ns ? __ldcg(p.ws_lse + (base + lane) * G + g) : -INFINITY;
        const float ls2 =
            g == warp ? ls_first_hi : lane + 32 < ns ? __ldcg(p.ws_lse + (base + lane + 32) * G + g) : -INFINITY;
        const bool nan = __any_sync(kFull, isnan(ls) || isnan(ls2));
        float M = fmaxf(ls, ls2);
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, x));
        const float e = M != -INFINITY && lane < ns ? exp2f(ls - M) : 0.f;
        const float e2 = M != -INFINITY && lane + 32 < ns ? exp2f(ls2 - M) : 0.f;
        float wsum = e + e2;
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) wsum += __shfl_xor_sync(kFull, wsum, x);
        const float inv = M != -INFINITY ? 1.f / wsum : 0.f;
        if (lane < ns) w[lane * G + g] = e * inv;
        if (lane + 32 < ns) w[(lane + 32) * G + g] = e2 * inv;
        if (lane == 0) {
            sm.merge_nan_h[g] = nan ? 1 : 0;
            const float lse2 = M != -INFINITY ? M + log2f(wsum) : -INFINITY;
            p.lse[static_cast<size_t>(b) * p.Hq + kvh * G + g] = nan ? NAN : lse2 * kLn2;
        }
    }
    cp_async_commit_wait_all();
    __syncthreads();   // every thread's copies and the weights visible
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    const float* ob = obuf + g_out * D + d;
#pragma unroll 2
    for (int s = part; s < ns; s += T) {
        const float ws = w[s * G + g_out];
        const float4 o = *reinterpret_cast<const float4*>(ob + s * G * D);
        acc.x = fmaf(ws, o.x, acc.x);
        acc.y = fmaf(ws, o.y, acc.y);
        acc.z = fmaf(ws, o.z, acc.z);
        acc.w = fmaf(ws, o.w, acc.w);
    }
#pragma unroll
    for (int x = W; x < 32; x <<= 1) {
        acc.x += __shfl_xor_sync(kFull, acc.x, x);
        acc.y += __shfl_xor_sync(kFull, acc.y, x);
        acc.z += __shfl_xor_sync(kFull, acc.z, x);
        acc.w += __shfl_xor_sync(kFull, acc.w, x);
    }
    if (part == 0)
        *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(b) * p.Hq + kvh * G + g_out) * D + d) =
            sm.merge_nan_h[g_out] ? make_float4(NAN, NAN, NAN, NAN) : acc;
    // A later TMA into the stages is ordered after the copies above; every
    // caller that reuses the stages passes a CTA barrier before it does.
    fence_proxy_async_shared();
}

// The fused merge of the last-arriving CTA for more splits than one pass
// holds (MergeCfg::kMaxSplits).  The ns partial outputs of (b, kvh) are
// contiguous in the workspace: every thread copies its share of
// them into the CTA's idle stage buffers with 16-byte cp.async (all in flight
// at once, a chunk of splits at a time), while the LSEs come in with plain L2
// loads; the weighted sum then runs out of shared memory, one float4 of the
// output per thread with independent loads.  Same arithmetic as merge_unit;
// all CTA threads call it.
template <int D, int G>
__device__ void merge_unit_staged(Smem<D, G>& sm, const AttnParams& p, int b, int kvh, int ns, int base_slot) {
    constexpr int kScratch = Cfg<D, G>::kStages * Cfg<D, G>::kMatBytes * 2;   // K and V stages
    constexpr int kSplitBytes = G * D * 4;
    constexpr int kOut = G * D / 4;                                            // float4 outputs of (b, kvh)
    constexpr int kPer = (kOut + kThreads - 1) / kThreads;
    const int tid = threadIdx.x;
    const size_t base = static_cast<size_t>(base_slot);
    uint8_t* scratch = &sm.k[0][0];   // k and v stages are adjacent
    float* w = reinterpret_cast<float*>(scratch);                  // [ns][G] weights
    const int w_bytes = (ns * G * 4 + 1023) & ~1023;
    float* obuf = reinterpret_cast<float*>(scratch + w_bytes);     // [chunk][G][D] partials
    const int chunk = (kScratch - w_bytes) / kSplitBytes;

    auto issue = [&](int s0) {   // every thread: its 16-byte pieces of splits [s0, s0 + chunk)
        const int vecs = min(chunk, ns - s0) * (kSplitBytes / 16);
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.ws_o + (base + s0) * G * D);
        const uint32_t dst = smem_addr(obuf);
        for (int i = tid; i < vecs; i += kThreads) cp_async16_plain(dst + i * 16, src + static_cast<size_t>(i) * 16);
    };
    const int warp = tid / 32, lane = tid % 32;
    issue(0);
    for (int i = tid; i < ns * G; i += kThreads) w[i] = __ldcg(p.ws_lse + base * G + i);
    __syncthreads();
    // per head: max and sum over the splits, one warp per head
    for (int g = warp; g < G; g += kThreads / 32) {
        float M = -INFINITY;
        bool nan = false;
        for (int s = lane; s < ns; s += 32) {
            nan |= isnan(w[s * G + g]);
            M = fmaxf(M, w[s * G + g]);
        }
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, x));
        nan = __any_sync(kFull, nan);
        float wsum = 0.f;
        if (M != -INFINITY)
            for (int s = lane; s < ns; s += 32) wsum += exp2f(w[s * G + g] - M);
#pragma unroll
        for (int x = 16; x > 0; x >>= 1) wsum += __shfl_xor_sync(kFull, wsum, x);
        if (lane == 0) {
            sm.merge_m[g] = M;
            sm.merge_inv[g] = M != -INFINITY ? 1.f / wsum : 0.f;
            sm.merge_nan_h[g] = nan ? 1 : 0;
            const float lse2 = M != -INFINITY ? M + log2f(wsum) : -INFINITY;
            p.lse[static_cast<size_t>(b) * p.Hq + kvh * G + g] = nan ? NAN : lse2 * kLn2;
        }
    }
    __syncthreads();
    for (int i = tid; i < ns * G; i += kThreads) {
        const int g = i % G;
        w[i] = sm.merge_m[g] != -INFINITY ? exp2f(w[i] - sm.merge_m[g]) * sm.merge_inv[g] : 0.f;
    }
    float4 acc[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = 0; s0 < ns; s0 += chunk) {
        const int n = min(chunk, ns - s0);
        cp_async_commit_wait_all();
        __syncthreads();   // this chunk (and the weights) visible to every thread
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const int i = tid + r * kThreads;
            if (i < kOut) {
                const int g = i / (D / 4), d = (i % (D / 4)) * 4;
                const float* wg = w + s0 * G + g;
                const float* og = obuf + g * D + d;
#pragma unroll 8
                for (int s = 0; s < n; ++s) {
                    const float ws = wg[s * G];
                    const float4 o = *reinterpret_cast<const float4*>(og + s * G * D);
                    acc[r].x = fmaf(ws, o.x, acc[r].x);
                    acc[r].y = fmaf(ws, o.y, acc[r].y);
                    acc[r].z = fmaf(ws, o.z, acc[r].z);
                    acc[r].w = fmaf(ws, o.w, acc[r].w);
                }
            }
        }
        if (s0 + chunk < ns) {
            __syncthreads();   // chunk consumed before it is overwritten
            issue(s0 + chunk);
        }
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int i = tid + r * kThreads;
        if (i < kOut) {
            const int g = i / (D / 4), d = (i % (D / 4)) * 4;
            *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(b) * p.Hq + kvh * G + g) * D + d) =
                sm.merge_nan_h[g] ? make_float4(NAN, NAN, NAN, NAN) : acc[r];
        }
    }
    // A later TMA into these stages is ordered after the copies above; every
    // caller that reuses the stages passes a CTA barrier before it does.
    fence_proxy_async_shared();
}

// ------------------------------------------------------------------ tile

// Tile of a queue entry: only the entry itself, so the producers can start
// streaming its planned pages at once (all of them are in the row's table).
__device__ __forceinline__ TileWork tile_from_item(const AttnParams& p, const pkv_work_item& it) {
    TileWork tw;
    tw.b = it.b;
    tw.kvh = it.kvh;
    tw.split = it.split;
    tw.page_begin = it.page_begin;
    tw.page_end = it.page_end;
    tw.t0 = it.page_begin * p.page_size;
    tw.t_stream = it.page_end * p.page_size;
    tw.t1 = tw.t_stream;
    tw.slot = 0;
    tw.finalize = 0;
    tw.splits = 0;
    tw.poisoned = 0;
    tw.lazy = 1;
    return tw;
}

// The rest of a queue tile: the row's length clips the token range, and the
// plan is checked against it (a mismatch poisons the tile and flags it).
__device__ __forceinline__ void tile_finish(const AttnParams& p, TileWork& tw) {
    const int n = p.seq_lens[tw.b];
    const int pages = (n + p.page_size - 1) / p.page_size;
    tw.splits = p.row_splits[tw.b];
    const int want_end = min((tw.split + 1) * p.chunk_pages, pages);
    tw.poisoned = (tw.page_begin != tw.split * p.chunk_pages || tw.page_end != want_end) ? 1 : 0;
    if (tw.poisoned && threadIdx.x == 0) atomicOr(&p.ctr->status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
    tw.t1 = tw.poisoned ? tw.t0 : min(tw.t_stream, n);
    tw.finalize = tw.splits == 1;
    tw.slot = p.row_start[tw.b] + tw.kvh * tw.splits + tw.split;
    tw.lazy = 0;
}

// One tile: the producer warp streams blocks, the consumer warps reduce them,
// then the four warp states are merged and written (to out/lse, or to the
// workspace for a split).  `pipe` counts blocks this CTA has streamed before
// (stage/phase bookkeeping continues across the tiles of a persistent CTA).
template <int D, int G, bool MMA>
__device__ void run_tile(Smem<D, G>& sm, const AttnParams& p, TileWork tw, uint32_t pipe,
                         const CUtensorMap* kmap, const CUtensorMap* vmap) {
    using C = Cfg<D, G>;
    constexpr int kStages = C::kStages;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int nblk = stream_blocks(tw);
    uint32_t* status = &p.ctr->status;

    if (warp >= kConsumerWarps) {
        // ---------------- producers
        if (nblk == 0) return;
        const int pw = warp - kConsumerWarps;
        const int ps = p.page_size;
        const int first_page = tw.t0 / ps;
        const int last_page = (tw.t_stream + ps - 1) / ps;   // exclusive
        const int32_t* bt_row = p.block_table + static_cast<size_t>(tw.b) * p.max_pages;
        const uint64_t policy = l2_evict_first_policy();
        const int bpp = ps / kBlockRows;   // blocks per page (page sizes are multiples of 16)
        int next_id = first_page + lane < last_page ? __ldg(bt_row + first_page + lane) : 0;
        for (int pg0 = first_page; pg0 < last_page; pg0 += 32) {
            const int ids = next_id;   // lane l: the table entry of page pg0 + l
            const int pg_next = pg0 + 32 + lane;
            next_id = pg_next < last_page ? __ldg(bt_row + pg_next) : 0;
            const int n_here = min(32, last_page - pg0);
            // Every lane checks its own entry once, and a batch with an entry outside
            // the pool is reported once; a block of such a page is not copied.
            if (__any_sync(kFull, lane < n_here && (ids < 0 || ids >= p.num_pages)) && lane == 0)
                atomicOr(status, static_cast<uint32_t>(PKV_DEV_PAGE_OOB));
            const int jb0 = (pg0 - first_page) * bpp;                     // the batch's blocks: [jb0, jb1)
            const int jb1 = min(nblk, (pg0 + n_here - first_page) * bpp);
            // this warp's blocks are j = pw (mod kProducerWarps)
            int j = jb0 + (pw - jb0 % kProducerWarps + kProducerWarps) % kProducerWarps;
            for (; j < jb1; j += kProducerWarps) {
                // the page's lane in the batch (one block per page for 16-token pages)
                const int pi = bpp == 1 ? j - jb0 : j / bpp - (pg0 - first_page);
                const int page = __shfl_sync(kFull, ids, pi);
                const int tok = tw.t0 + j * kBlockRows;
                const int page_tok0 = (pg0 + pi) * ps;
                const bool page_ok = (page >= 0) & (page < p.num_pages);
                const uint32_t it = pipe + j;
                const int s = it % kStages;
                const uint32_t use = it / kStages;
                int go = 0;
                if (lane == 0) {
                    go = !sm.abort;
                    if (go && use > 0) go = mbar_wait(&sm.empty[s], (use - 1) & 1u, status, &sm.abort);
                    go &= page_ok;
                    sm.bad[s] = !go;
                    if (go) sm.issued[s] = use + 1;
                    if (p.copy_lsu)
                        mbar_arrive(&sm.full[s]);   // publishes bad[s]; the lanes' copies arrive below
                    else if (go)
                        mbar_arrive_expect_tx(&sm.full[s], C::kStageBytes);
                    else
                        mbar_arrive(&sm.full[s]);
                }
                go = __shfl_sync(kFull, go, 0);
                const int grow = page * ps + (tok - page_tok0);   // token row inside the pool
                if (p.copy_lsu) {
                    // every lane moves D/16 16-byte chunks of K and as many of V
                    // into the swizzled stage, then arrives when they have landed
                    if (go) {
                        const size_t row0 = (static_cast<size_t>(grow) * p.Hkv + tw.kvh) * D;
                        const size_t pitch = static_cast<size_t>(p.Hkv) * D;
                        const uint32_t ks = smem_addr(sm.k[s]), vs = smem_addr(sm.v[s]);
#pragma unroll
                        for (int i = 0; i < kBlockRows * (D / 8) / 32; ++i) {
                            const int q = lane + 32 * i;
                            const int r = q / (D / 8), c = (q % (D / 8)) * 8;
                            const size_t off = row0 + r * pitch + c;
                            cp_async16(ks + swz(r, c), p.k_pages + off, policy);
                            cp_async16(vs + swz(r, c), p.v_pages + off, policy);
                        }
                    }
                    cp_async_arrive_noinc(&sm.full[s]);
                } else if (go && lane < 2 * (D / 64)) {
                    // the block's D/64 K boxes and D/64 V boxes, after lane 0 armed the barrier
                    const int h = lane % (D / 64);
                    const bool is_v = lane >= D / 64;
                    tma_load_3d((is_v ? sm.v[s] : sm.k[s]) + h * (kBlockRows * 128), is_v ? vmap : kmap, h * 64,
                                tw.kvh, grow, &sm.full[s], policy);
                }
            }
        }
        return;
    }

    // ---------------- consumers
    // (queue tiles: the lengths and row table are read here, while the producers
    // already stream the planned pages)
    if (tw.lazy) tile_finish(p, tw);
    if (threadIdx.x == 0) {
        sm.tile_fin = tw.finalize;
        sm.tile_splits = tw.splits;
        sm.tile_base = tw.slot - tw.split;   // the merge needs no second read of the row table
    }
    const int ntok = tw.t1 > tw.t0 ? tw.t1 - tw.t0 : 0;
    int poisoned = tw.poisoned;
    if constexpr (MMA) {
        MmaState<D, G> st;
        mma_init<D, G>(st, p, tw, lane);
        for (int j = warp; j < nblk; j += kConsumerWarps) {
            const uint32_t it = pipe + j;
            const int s = it % kStages;
            const bool ok = mbar_wait(&sm.full[s], (it / kStages) & 1u, status, &sm.abort);
            if (p.trace && threadIdx.x == 0 && sm.tr[kTrFirstBlock] == 0) sm.tr[kTrFirstBlock] = globaltimer_ns();
            const int valid = min(kBlockRows, ntok - j * kBlockRows);
            if (!ok || sm.bad[s] || valid <= 0) {   // nothing to reduce (or past the row's end)
                if (!ok || sm.bad[s]) poisoned = 1;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[s]);
            } else {   // releases the stage itself once the block is in registers
                mma_block<D, G>(st, sm.k[s], sm.v[s], &sm.empty[s], sm.pt[warp], valid, lane, p.scale_log2);
            }
        }
        trace_stamp(sm, p, kTrStreamEnd);
        mma_publish<D, G>(st, sm, warp, lane);
    } else {
        FmaState<D, G> st;
        fma_init<D, G>(st, p, tw, lane);
        for (int j = warp; j < nblk; j += kConsumerWarps) {
            const uint32_t it = pipe + j;
            const int s = it % kStages;
            const bool ok = mbar_wait(&sm.full[s], (it / kStages) & 1u, status, &sm.abort);
            if (p.trace && threadIdx.x == 0 && sm.tr[kTrFirstBlock] == 0) sm.tr[kTrFirstBlock] = globaltimer_ns();
            const int valid = min(kBlockRows, ntok - j * kBlockRows);
            if (!ok || sm.bad[s])
                poisoned = 1;
            else if (valid > 0)
                fma_block<D, G>(st, sm.k[s], sm.v[s], sm.p[warp], valid, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
        trace_stamp(sm, p, kTrStreamEnd);
        fma_publish<D, G>(st, sm, warp, lane);
    }
    if (lane == 0) sm.poisoned[warp] = poisoned;
    named_barrier_sync(1, kConsumerWarps * 32);

    // Exact LSE combine of the four warp states: one float4 (head g, d .. d+3)
    // per thread and pass, so every thread runs one short independent chain.
    const int tid = threadIdx.x;
    bool any_poison = false;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) any_poison |= sm.poisoned[w] != 0;
    constexpr int kItems = G * D / 4;
    for (int i = tid; i < kItems; i += kConsumerWarps * 32) {
        const int g = i / (D / 4), d = (i % (D / 4)) * 4;
        float mw[kConsumerWarps];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
            mw[w] = sm.m[w][g];
            M = fmaxf(M, mw[w]);
        }
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse2 = -INFINITY;
        if (M != -INFINITY) {
            float lsum = 0.f;
            float4 os = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float sc = exp2f(mw[w] - M);   // idle warp: m = -inf -> 0
                lsum = fmaf(sm.l[w][g], sc, lsum);
                const float4 a = *reinterpret_cast<const float4*>(&sm.acc[w][g * D + d]);
                os.x = fmaf(a.x, sc, os.x);
                os.y = fmaf(a.y, sc, os.y);
                os.z = fmaf(a.z, sc, os.z);
                os.w = fmaf(a.w, sc, os.w);
            }
            const float inv = 1.f / lsum;
            o = make_float4(os.x * inv, os.y * inv, os.z * inv, os.w * inv);
            lse2 = M + log2f(lsum);
        }
        if (any_poison) {
            o = make_float4(NAN, NAN, NAN, NAN);
            lse2 = NAN;
        }
        if (tw.finalize) {
            const int h = tw.kvh * G + g;
            *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(tw.b) * p.Hq + h) * D + d) = o;
            if (d == 0) p.lse[static_cast<size_t>(tw.b) * p.Hq + h] = lse2 * kLn2;
        } else {
            *reinterpret_cast<float4*>(p.ws_o + (static_cast<size_t>(tw.slot) * G + g) * D + d) = o;
            if (d == 0) p.ws_lse[static_cast<size_t>(tw.slot) * G + g] = lse2;
        }
    }
    if (p.trace && threadIdx.x == 0) {
        sm.tr[kTrCombineEnd] = globaltimer_ns();
        sm.tr[kTrLastTile] = (static_cast<uint64_t>(tw.b) << 40) | (static_cast<uint64_t>(tw.kvh) << 20) |
                             static_cast<uint64_t>(tw.split);
        sm.tr[kTrTiles] += 1;
    }
}

// After a split tile has written its partial: the last split of (b, kvh) to
// arrive merges all of them (all CTA threads call this).
template <int D, int G>
__device__ void merge_if_last(Smem<D, G>& sm, const AttnParams& p, int b, int kvh, int ns) {
    // The CTA's partial is written; after the barrier, thread 0's fence makes those
    // writes visible device-wide before its arrival is counted (release), and the
    // arrival's acquire orders the other splits' writes before our reads.  The
    // counter's reset needs no fence: the next launch reads it only after this grid
    // has completed.  (The caller has just passed a barrier too; dropping this one
    // measured slower.)
    __syncthreads();
    if (threadIdx.x == 0) {
        const int u = b * p.Hkv + kvh;
        fence_acq_rel_gpu();
        const uint32_t prev = atom_add_acquire_gpu(&p.arrive[u], 1u);
        const int last = prev == static_cast<uint32_t>(ns - 1);
        if (last) p.arrive[u] = 0;   // ready for the next launch
        sm.tile_slot[1] = last;
        if (p.trace) sm.tr[kTrArrived] = globaltimer_ns();
    }
    __syncthreads();
    if (sm.tile_slot[1]) {
        // the stage buffers are idle here and serve as the merge's scratch
        static_assert(2 * Cfg<D, G>::kStages * Cfg<D, G>::kMatBytes >= kMergeCapFloats * 4 + 2 * G * D * 4,
                      "merge scratch");
        if (ns <= MergeCfg<D, G>::kMaxSplits)
            merge_unit_onepass<D, G>(sm, p, b, kvh, ns, sm.tile_base);
        else
            merge_unit_staged<D, G>(sm, p, b, kvh, ns, sm.tile_base);
        trace_stamp(sm, p, kTrMergeEnd);
    }
}

// The merge shared by all ns splits of (b, kvh), for a launch whose CTAs are
// all resident at once (cooperative launch of one wave).  Each split publishes
// its partial, waits until all ns have arrived, then merges its own 1/ns share
// of the G*D/4 float4 outputs, lanes over the splits, so each CTA reads only
// its share's columns of every partial (plus the LSEs) instead of one CTA
// reading all of them.  Every split departs once after the
// wait; the last to depart rewinds both counters for the next launch.  Same
// exact LSE rule as merge_unit (all CTA threads call this).
template <int D, int G>
__device__ void merge_all_splits(Smem<D, G>& sm, const AttnParams& p, int b, int kvh, int split, int ns) {
    __syncthreads();
    const int u = b * p.Hkv + kvh;
    uint32_t* arrive = p.arrive + u;
    uint32_t* depart = p.arrive + static_cast<size_t>(p.B) * p.Hkv + u;
    uint32_t departed = 0;   // thread 0: departures before this one (read after the merge)
    if (threadIdx.x == 0) {
        fence_acq_rel_gpu();   // release: the partial written above, before the arrival
        atomicAdd(arrive, 1u);
        const bool ok = wait_count(arrive, static_cast<uint32_t>(ns), &p.ctr->status, &sm.abort);
        departed = atomicAdd(depart, 1u);
        sm.tile_slot[1] = ok;
        if (p.trace) sm.tr[kTrArrived] = globaltimer_ns();
    }
    __syncthreads();
    const bool ok = sm.tile_slot[1] != 0;
    // This split's share: float4 outputs [i0, i1).  L lanes (a power of two, at
    // most 32, at least ns when ns <= 32) merge one output over the splits, so
    // a warp covers 32 / L outputs per pass and the whole share usually takes
    // one pass: every load of the share is in flight at once.
    constexpr int kItems = G * D / 4;
    const int per = (kItems + ns - 1) / ns;
    const int i0 = split * per, i1 = min(kItems, i0 + per);
    int L = 1;
    while (L < ns && L < 32) L <<= 1;
    const int groups = 32 / L;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int sub = lane % L, grp = lane / L;
    const size_t base = static_cast<size_t>(sm.tile_base);
    for (int pass = i0; pass < i1; pass += (kThreads / 32) * groups) {   // uniform over the CTA
        const int i = pass + warp * groups + grp;
        const bool live = i < i1;
        const int g = live ? i / (D / 4) : 0, d = live ? (i % (D / 4)) * 4 : 0;
        float m = -INFINITY, l = 0.f;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        int nan = 0;
        if (live) {
            for (int s = sub; s < ns; s += L) {   // the lane's splits, merged online
                const float ls = __ldcg(p.ws_lse + (base + s) * G + g);
                const float4 o = __ldcg(reinterpret_cast<const float4*>(p.ws_o + ((base + s) * G + g) * D + d));
                nan |= isnan(ls) ? 1 : 0;
                if (ls > m) {
                    const float c = exp2f(m - ls);   // m = -inf: 0
                    l *= c;
                    a.x *= c;
                    a.y *= c;
                    a.z *= c;
                    a.w *= c;
                    m = ls;
                }
                if (ls != -INFINITY) {
                    const float e = exp2f(ls - m);
                    l += e;
                    a.x = fmaf(e, o.x, a.x);
                    a.y = fmaf(e, o.y, a.y);
                    a.z = fmaf(e, o.z, a.z);
                    a.w = fmaf(e, o.w, a.w);
                }
            }
        }
        // combine the L lanes of the group (xor partners stay inside it)
        float M = m;
        for (int x = L / 2; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, x));
        const float sc = m != -INFINITY ? exp2f(m - M) : 0.f;
        l *= sc;
        a.x *= sc;
        a.y *= sc;
        a.z *= sc;
        a.w *= sc;
        for (int x = L / 2; x > 0; x >>= 1) {
            l += __shfl_xor_sync(kFull, l, x);
            a.x += __shfl_xor_sync(kFull, a.x, x);
            a.y += __shfl_xor_sync(kFull, a.y, x);
            a.z += __shfl_xor_sync(kFull, a.z, x);
            a.w += __shfl_xor_sync(kFull, a.w, x);
            nan |= __shfl_xor_sync(kFull, nan, x);
        }
        if (live && sub == 0) {
            float4 o;
            float lse2;
            if (nan || !ok) {
                o = make_float4(NAN, NAN, NAN, NAN);
                lse2 = NAN;
            } else if (M == -INFINITY) {
                o = make_float4(0.f, 0.f, 0.f, 0.f);
                lse2 = -INFINITY;
            } else {
                const float inv = 1.f / l;
                o = make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv);
                lse2 = M + log2f(l);
            }
            const int h = kvh * G + g;
            *reinterpret_cast<float4*>(p.out + (static_cast<size_t>(b) * p.Hq + h) * D + d) = o;
            if (d == 0) p.lse[static_cast<size_t>(b) * p.Hq + h] = lse2 * kLn2;
        }
    }
    if (threadIdx.x == 0 && departed == static_cast<uint32_t>(ns - 1)) {
        *arrive = 0;   // every split has seen the full count: ready for the next launch
        *depart = 0;
    }
}

// After an abort, wait (bounded again) for every TMA copy this CTA issued, so
// that none lands in shared memory after the CTA has moved on or exited.
// Called by one thread once the producer has stopped issuing.
template <int D, int G>
__device__ void drain_after_abort(Smem<D, G>& sm, uint32_t* status) {
    for (int s = 0; s < Cfg<D, G>::kStages; ++s)
        if (sm.issued[s] > 0) mbar_wait_slow(&sm.full[s], (sm.issued[s] - 1) & 1u, status, nullptr);
}

template <int D, int G, bool MMA>
__global__ void __launch_bounds__(kThreads, MMA ? 2 : 1) attention_kernel(const AttnParams p,
                                                             const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ uint8_t smem_raw[];
    Smem<D, G>& sm =
        *reinterpret_cast<Smem<D, G>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    if (p.trace && threadIdx.x == 0) {
        for (int i = 0; i < kTraceWords; ++i) sm.tr[i] = 0;
        sm.tr[kTrEntry] = globaltimer_ns();
        sm.tr[kTrSm] = smid();
    }
    // Before the grid dependency wait, only data no kernel writes may be used:
    // the host-staged queue entry.  The producers also warm L2 with the first
    // ring's worth of the tile's K/V rows, reading the block table
    // speculatively: prefetches change no value, and every value used below is
    // read again after the wait.
    const bool staged_item = p.route == kRouteQueue && p.queue_host_staged && static_cast<int>(blockIdx.x) < p.num_tiles;
    pkv_work_item item{};
    if (staged_item) {
        item = p.queue[blockIdx.x];
        const int pw = static_cast<int>(threadIdx.x) / 32 - kConsumerWarps;
        if (pw >= 0 && item.b >= 0 && item.b < p.B && item.kvh >= 0 && item.kvh < p.Hkv && item.page_begin >= 0 &&
            item.page_end <= p.max_pages) {
            const int lane = threadIdx.x % 32;
            const int ps = p.page_size;
            const int t0 = item.page_begin * ps;
            const int t_end = min(item.page_end * ps, t0 + kPrefetchBlocks * kBlockRows);
            const int32_t* bt_row = p.block_table + static_cast<size_t>(item.b) * p.max_pages;
            for (int tok = t0 + pw * 32 + lane; tok < t_end; tok += kProducerWarps * 32) {
                const int page = ld_volatile_i32(bt_row + tok / ps);
                if (page < 0 || page >= p.num_pages) continue;
                const size_t row = (static_cast<size_t>(page) * ps + tok % ps) * p.Hkv + item.kvh;
#pragma unroll
                for (int c = 0; c < D * 2; c += 128) {
                    prefetch_l2(reinterpret_cast<const uint8_t*>(p.k_pages + row * D) + c);
                    prefetch_l2(reinterpret_cast<const uint8_t*>(p.v_pages + row * D) + c);
                }
            }
        }
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg<D, G>::kStages; ++s) {
            // LSU copies: 32 producer lanes' cp.async arrivals + lane 0's flag arrival
            mbar_init(&sm.full[s], p.copy_lsu ? 33 : 1);
            mbar_init(&sm.empty[s], 1);
            sm.issued[s] = 0;
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    // Everything below reads what earlier kernels in the stream may have
    // written (q, pages, lengths, table, plan): wait for them first.
    grid_dependency_wait();
    trace_stamp(sm, p, kTrWaitDone);
    __syncthreads();
    // the CTA's timeline row goes out once the CTA is done (after the wait, so
    // an overlapping earlier launch has finished with the same row)
    auto trace_flush = [&]() {
        if (p.trace && threadIdx.x == 0) {
            sm.tr[kTrExit] = globaltimer_ns();
            uint64_t* row = p.trace + static_cast<size_t>(blockIdx.x) * kTraceWords;
            for (int i = 0; i < kTraceWords; ++i) row[i] = sm.tr[i];
        }
    };
    // rows with no tokens get no tiles: their neutral state is written after
    // the CTA's own tile, off the tile's critical path
    auto neutral_rows = [&]() {
        if (p.no_empty_rows) return;   // the plan has no empty row
        for (int b = blockIdx.x; b < p.B; b += gridDim.x)
            if (p.row_splits[b] == 0) write_neutral_row(p, b, threadIdx.x, blockDim.x);
    };

    if (p.route == kRoutePersistent) {
        const int num_tiles = p.tiles_d ? *p.tiles_d : p.num_tiles;   // a device-planned step sets it
        uint32_t pipe = 0;
        while (true) {
            if (threadIdx.x == 0) sm.tile_slot[0] = static_cast<int>(atomicAdd(&p.ctr->next_tile, 1u));
            __syncthreads();
            const int t = sm.tile_slot[0];
            if (t >= num_tiles) break;
            const TileWork tw = tile_from_item(p, p.queue[p.order ? p.order[t] : t]);
            run_tile<D, G, MMA>(sm, p, tw, pipe, &kmap, &vmap);
            pipe += stream_blocks(tw);
            __syncthreads();
            if (!sm.tile_fin && p.fused_merge) merge_if_last<D, G>(sm, p, tw.b, tw.kvh, sm.tile_splits);
            __syncthreads();
        }
        launch_dependents();
        neutral_rows();
        if (threadIdx.x == 0) {
            if (sm.abort) drain_after_abort<D, G>(sm, &p.ctr->status);
            // the last CTA out rewinds the queue for the next launch
            if (atomicAdd(&p.ctr->done_ctas, 1u) == gridDim.x - 1) {
                p.ctr->next_tile = 0;
                p.ctr->done_ctas = 0;
            }
        }
        trace_flush();
        return;
    }

    TileWork tw;
    tw.lazy = 0;
    tw.split = tw.page_begin = tw.page_end = 0;
    if (p.route == kRouteDirect) {
        tw.b = blockIdx.x / p.Hkv;
        tw.kvh = blockIdx.x % p.Hkv;
        tw.t0 = 0;
        tw.t1 = p.seq_lens[tw.b];
        tw.slot = 0;
        tw.finalize = 1;
        tw.splits = 1;
        tw.poisoned = 0;
        if (tw.t1 < 0 || tw.t1 > p.max_pages * p.page_size) {   // would read past the table row
            tw.poisoned = 1;
            tw.t1 = 0;
            if (threadIdx.x == 0) atomicOr(&p.ctr->status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
        }
        tw.t_stream = tw.t1;
    } else if (p.route == kRouteQueue) {
        if (static_cast<int>(blockIdx.x) >= p.num_tiles) {   // launched only for the neutral rows
            launch_dependents();
            neutral_rows();
            trace_flush();
            return;
        }
        tw = tile_from_item(p, staged_item ? item : p.queue[blockIdx.x]);
    } else {   // padded grid: (b, kvh, s) from the block index, ranges from the device lengths
        const int per_row = p.Hkv * p.max_splits;
        tw.b = blockIdx.x / per_row;
        tw.kvh = (blockIdx.x % per_row) / p.max_splits;
        const int s = blockIdx.x % p.max_splits;
        tw.split = s;
        const int n = p.seq_lens[tw.b];
        const int pages = (n + p.page_size - 1) / p.page_size;
        tw.poisoned = n < 0 || pages > p.max_splits * p.chunk_pages || n > p.max_pages * p.page_size;
        if (tw.poisoned && threadIdx.x == 0) atomicOr(&p.ctr->status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
        const int pb = max(0, min(s * p.chunk_pages, pages));
        const int pe = max(0, min((s + 1) * p.chunk_pages, pages));
        tw.t0 = pb * p.page_size;
        tw.t1 = tw.poisoned ? tw.t0 : min(pe * p.page_size, n);
        tw.t_stream = tw.t1;
        tw.finalize = p.max_splits == 1;
        tw.splits = p.max_splits;
        tw.slot = blockIdx.x;
    }
    run_tile<D, G, MMA>(sm, p, tw, 0, &kmap, &vmap);
    __syncthreads();
    launch_dependents();   // the next grid may start its CTAs in the slots this tail frees
    if (!sm.tile_fin && p.fused_merge) {
        if (p.all_merge)
            merge_all_splits<D, G>(sm, p, tw.b, tw.kvh, tw.split, sm.tile_splits);
        else
            merge_if_last<D, G>(sm, p, tw.b, tw.kvh, sm.tile_splits);
    }
    if (p.route == kRouteQueue) neutral_rows();
    if (threadIdx.x == 0 && sm.abort) drain_after_abort<D, G>(sm, &p.ctr->status);
    trace_flush();
}

// ------------------------------------------------------------------ resident steps
//
// One cooperative launch that stays resident across continuous-decoding steps,
// as the persistent worker of "GPUOS" (arXiv 2604.17861, section 4.1) and the
// resident beat of "WPK persistent kernel" (dotwave.ai) do.  Per step:
//   CTA 0 waits (bounded) for the host to publish the step in the mapped
//   control block, applies its slot requests, then allocates pages and builds
//   the plan (the device planner of pkv_devplan.cuh) -- grid barrier -- every
//   CTA appends the new tokens of its rows and marks each row ready (a release
//   store of the step number) -- the CTAs drain the step's queue as the
//   persistent route does (fused last-arriver merge), each tile first waiting
//   (acquire, bounded) until its row is marked ready -- the last CTA to finish
//   publishes the step's outputs to the host (system-scope release).  One grid
//   barrier per step; a step that admits new sessions also has one after the
//   prompt copy, which every CTA shares.  The host publishes the next step only
//   after this one, so the next plan never overwrites a queue still in use.
// With yield_every > 0 the kernel leaves the GPU after that many steps (exited =
// 3), so that a long session does not hold every SM; the host relaunches it.
// Every wait is bounded: the host wait by idle_limit_ns, a grid barrier by
// kWaitLimitNs; on expiry the status word gets PKV_DEV_TIMEOUT, the abort word
// is raised and every CTA leaves the loop at its next barrier.

enum ResidentCmd : uint32_t { kCmdGo = 1, kCmdStop = 2, kCmdFail = 3 };

// Grid barrier of a cooperative launch (all CTAs resident).  Returns false if
// the barrier was aborted or ran out of time.
template <int D, int G>
__device__ bool grid_barrier(Smem<D, G>& sm, uint32_t* gs, uint32_t* status, uint64_t limit_ns = kWaitLimitNs) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        if (*reinterpret_cast<volatile uint32_t*>(gs + kSyncAbort)) {
            ok = 0;
        } else {
            const uint32_t gen = ld_acquire_gpu(gs + kSyncGen);
            fence_acq_rel_gpu();   // this CTA's writes before its arrival
            if (atomicAdd(gs + kSyncCount, 1u) == gridDim.x - 1) {
                gs[kSyncCount] = 0;
                st_release_gpu(gs + kSyncGen, gen + 1);
            } else {
                const uint64_t t0 = globaltimer_ns();
                while (ld_acquire_gpu(gs + kSyncGen) == gen) {
                    if (*reinterpret_cast<volatile uint32_t*>(gs + kSyncAbort)) {
                        ok = 0;
                        break;
                    }
                    if (globaltimer_ns() - t0 > limit_ns) {
                        atomicOr(status, static_cast<uint32_t>(PKV_DEV_TIMEOUT));
                        atomicExch(gs + kSyncAbort, 1u);
                        ok = 0;
                        break;
                    }
                    __nanosleep(64);
                }
            }
        }
        sm.sync_ok = ok;
    }
    __syncthreads();
    return sm.sync_ok != 0;
}

// CTA 0, thread 0: wait for the host to publish `step` (or to stop).
__device__ uint32_t wait_host_step(const ResidentCtl* ctl, uint32_t step, uint64_t limit_ns, uint32_t* status) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (ld_acquire_sys(&ctl->step) >= step) return kCmdGo;
        if (ld_acquire_sys(&ctl->stop)) return kCmdStop;
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, static_cast<uint32_t>(PKV_DEV_TIMEOUT));
            return kCmdFail;
        }
        __nanosleep(200);
    }
}

template <int D, int G, bool MMA>
__global__ void __launch_bounds__(kThreads, MMA ? 2 : 1) resident_kernel(const ResidentParams rp,
                                                                         const __grid_constant__ CUtensorMap kmap,
                                                                         const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ uint8_t smem_raw[];
    Smem<D, G>& sm =
        *reinterpret_cast<Smem<D, G>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const AttnParams& p = rp.attn;
    uint32_t* status = &p.ctr->status;
    uint32_t* gs = rp.grid_sync;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg<D, G>::kStages; ++s) {
            mbar_init(&sm.full[s], p.copy_lsu ? 33 : 1);
            mbar_init(&sm.empty[s], 1);
            sm.issued[s] = 0;
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    uint32_t pipe = 0;
    bool failed = false, yielded = false;
    for (uint32_t step = rp.first_step;; ++step) {
        // ---- 1. CTA 0: the host's step, then allocation and plan
        if (blockIdx.x == 0) {
            if (threadIdx.x == 0) {
                const uint32_t cmd = wait_host_step(rp.ctl, step, rp.idle_limit_ns, status);
                if (cmd == kCmdGo) {
                    p.ctr->next_tile = 0;
                    if (rp.times) rp.times[4 * ((step - 1) % rp.times_cap)] = globaltimer_ns();
                }
                if (cmd == kCmdFail) atomicExch(gs + kSyncAbort, 1u);
                gs[kSyncCmd] = cmd;
                sm.tile_slot[0] = static_cast<int>(cmd);
            }
            __syncthreads();
            if (sm.tile_slot[0] == kCmdGo) {
                // the step's slot requests (evictions, admissions) before its allocation and plan
                if (threadIdx.x == 0) {
                    const uint32_t n = min(*reinterpret_cast<volatile uint32_t*>(&rp.ctl->requests),
                                           static_cast<uint32_t>(PKV_RESIDENT_MAX_REQUESTS));
                    gs[kSyncReq] = n;
                    if (n) {
                        SlotParams sp = rp.slots;
                        sp.n = static_cast<int32_t>(n);
                        slots::apply_requests(sp);
                    }
                }
                __syncthreads();
                int* scratch = reinterpret_cast<int*>(&sm.k[0][0]);   // the idle ring (K and V stages)
                devplan::plan_step<kThreads>(rp.plan, scratch);
                fence_proxy_async_shared();   // generic writes to the ring before later TMA writes
            }
        }
        // (CTA 0 may wait up to idle_limit_ns for the host before it arrives)
        if (!grid_barrier<D, G>(sm, gs, status, rp.idle_limit_ns + kWaitLimitNs)) {
            failed = true;
            break;
        }
        if (*reinterpret_cast<volatile uint32_t*>(gs + kSyncCmd) != kCmdGo) break;
        if (blockIdx.x == 0 && threadIdx.x == 0 && rp.times) rp.times[4 * ((step - 1) % rp.times_cap) + 1] = globaltimer_ns();

        // ---- 2. the admitted rows' prompts, then the append: every CTA takes rows
        // blockIdx.x, blockIdx.x + gridDim.x, ... (idle slots are left alone)
        if (const int nreq = static_cast<int>(*reinterpret_cast<volatile uint32_t*>(gs + kSyncReq))) {
            SlotParams sp = rp.slots;
            sp.n = nreq;
            slots::copy_prompts(sp, static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x,
                                static_cast<int64_t>(gridDim.x) * kThreads);
        }
        for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
            if (rp.plan.active && !rp.plan.active[b]) continue;   // uniform over the CTA
            if (threadIdx.x == 0) {
                const int pos = rp.lens_w[b];
                int page = -1;
                if (pos < 0 || pos / p.page_size >= p.max_pages) {
                    atomicOr(status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));
                } else {
                    page = p.block_table[static_cast<size_t>(b) * p.max_pages + pos / p.page_size];
                    if (page < 0) {   // no page assigned for the new position
                        atomicOr(status, static_cast<uint32_t>(PKV_DEV_ROW_FULL));
                        page = -1;
                    } else if (page >= p.num_pages) {
                        atomicOr(status, static_cast<uint32_t>(PKV_DEV_PAGE_OOB));
                        page = -1;
                    }
                }
                sm.append_page = page;
                sm.append_pos = pos;
            }
            __syncthreads();
            if (sm.append_page >= 0) {
                const int row = p.Hkv * D;
                const size_t dst = (static_cast<size_t>(sm.append_page) * p.page_size + sm.append_pos % p.page_size) * row;
                const size_t src = static_cast<size_t>(b) * row;
                for (int c = threadIdx.x * 8; c < row; c += kThreads * 8) {
                    *reinterpret_cast<uint4*>(rp.k_pages_w + dst + c) = *reinterpret_cast<const uint4*>(rp.k_new + src + c);
                    *reinterpret_cast<uint4*>(rp.v_pages_w + dst + c) = *reinterpret_cast<const uint4*>(rp.v_new + src + c);
                }
                if (threadIdx.x == 0) rp.lens_w[b] = sm.append_pos + 1;
            }
            __syncthreads();   // the row's writes are done: mark it ready for the drain
            if (threadIdx.x == 0) st_release_gpu(rp.row_ready + b, step);
        }
        // admitted prompts are copied by every CTA: the drain waits for all of them
        const bool prompts = *reinterpret_cast<volatile uint32_t*>(gs + kSyncReq) != 0;
        if (prompts && !grid_barrier<D, G>(sm, gs, status)) {
            failed = true;
            break;
        }

        // ---- 3. decode: drain the step's queue (the persistent route)
        if (blockIdx.x == 0 && threadIdx.x == 0 && rp.times) rp.times[4 * ((step - 1) % rp.times_cap) + 2] = globaltimer_ns();
        const int num_tiles = *p.tiles_d;
        while (true) {
            if (threadIdx.x == 0) {
                const int t = static_cast<int>(atomicAdd(&p.ctr->next_tile, 1u));
                sm.tile_slot[0] = t;
                // the tile's row must have its new token (acquire of the appender's release)
                if (t < num_tiles && !prompts) {
                    const uint32_t* flag = rp.row_ready + p.queue[p.order[t]].b;
                    if (ld_acquire_gpu(flag) < step) wait_count(flag, step, status, &sm.abort);
                    if (!p.copy_lsu) fence_proxy_async_global();   // TMA reads what plain stores wrote
                }
            }
            __syncthreads();
            const int t = sm.tile_slot[0];
            if (t >= num_tiles) break;
            const TileWork tw = tile_from_item(p, p.queue[p.order[t]]);
            run_tile<D, G, MMA>(sm, p, tw, pipe, &kmap, &vmap);
            pipe += stream_blocks(tw);
            __syncthreads();
            if (!sm.tile_fin && p.fused_merge) merge_if_last<D, G>(sm, p, tw.b, tw.kvh, sm.tile_splits);
            __syncthreads();
        }
        for (int b = blockIdx.x; b < p.B; b += gridDim.x)
            if (p.row_splits[b] == 0) write_neutral_row(p, b, threadIdx.x, blockDim.x);
        if (sm.abort) atomicExch(gs + kSyncAbort, 1u);   // a bounded wait of this CTA ran out
        __syncthreads();   // this CTA's outputs of the step are written

        // ---- 4. the last CTA done publishes the step's outputs to the host
        if (threadIdx.x == 0) {
            fence_acq_rel_gpu();   // release this CTA's outputs before its count
            if (atomicAdd(gs + kSyncDone, 1u) == gridDim.x - 1) {
                fence_acq_rel_gpu();   // acquire every other CTA's outputs
                gs[kSyncDone] = 0;
                if (rp.times) rp.times[4 * ((step - 1) % rp.times_cap) + 3] = globaltimer_ns();
                fence_sc_sys();
                st_release_sys(&rp.ctl->done, step);
            }
        }
        if (rp.yield_every > 0 && (step - rp.first_step + 1) % static_cast<uint32_t>(rp.yield_every) == 0) {
            yielded = true;   // leave the GPU; the host relaunches for the next step
            break;
        }
    }
    if (threadIdx.x == 0 && sm.abort) drain_after_abort<D, G>(sm, status);
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        fence_sc_sys();
        st_release_sys(&rp.ctl->exited, failed ? 2u : yielded ? 3u : 1u);
    }
}

template <int D, int G, bool MMA>
cudaError_t launch_resident_t(const ResidentParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                              cudaStream_t stream) {
    constexpr size_t smem = smem_bytes<D, G>();
    static_assert(2 * Cfg<D, G>::kStages * Cfg<D, G>::kMatBytes >= devplan::kPlanScratchInts * 4, "planner scratch");
    cudaError_t e = cudaFuncSetAttribute(resident_kernel<D, G, MMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // the grid barriers need every CTA resident
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, resident_kernel<D, G, MMA>, p, kmap, vmap);
}

template <int D, int G, bool MMA>
int resident_ctas_per_sm_t() {
    constexpr size_t smem = smem_bytes<D, G>();
    if (cudaFuncSetAttribute(resident_kernel<D, G, MMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, resident_kernel<D, G, MMA>, kThreads, smem) != cudaSuccess)
        return 0;
    return n;
}

template <int D, int G>
__global__ void __launch_bounds__(128) merge_kernel(const AttnParams p) {
    __shared__ float wsm[kMergeCapFloats];
    __shared__ float m_s[G], inv_s[G];
    __shared__ int nan_s;
    const int b = blockIdx.x / p.Hkv;
    const int kvh = blockIdx.x % p.Hkv;
    const int ns = p.row_splits[b];
    if (ns == 1) return;   // that row's tile wrote out / lse itself
    if (ns == 0) {
        for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
            const int h = kvh * G + idx / D;
            p.out[(static_cast<size_t>(b) * p.Hq + h) * D + idx % D] = 0.f;
            if (idx % D == 0) p.lse[static_cast<size_t>(b) * p.Hq + h] = -INFINITY;
        }
        return;
    }
    merge_unit<D, G>(p, b, kvh, ns, wsm, m_s, inv_s, &nan_s);
}

template <int D, int G, bool MMA>
cudaError_t launch_attention_t(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                               cudaStream_t stream, bool cooperative) {
    constexpr size_t smem = smem_bytes<D, G>();
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attention_kernel<D, G, MMA>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    // The launch may overlap the tail of the previous kernel in the stream
    // (programmatic dependent launch; the kernel waits for it before reading
    // anything); cooperative: every CTA resident at once, or the launch fails.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cooperative) {
        attr[n].id = cudaLaunchAttributeCooperative;
        attr[n].val.cooperative = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, attention_kernel<D, G, MMA>, p, kmap, vmap);
}

template <int D, int G, bool MMA>
int ctas_per_sm_t() {
    constexpr size_t smem = smem_bytes<D, G>();
    if (cudaFuncSetAttribute(attention_kernel<D, G, MMA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attention_kernel<D, G, MMA>, kThreads, smem) !=
        cudaSuccess)
        return 0;
    return n;
}

template <int D, int G>
cudaError_t launch_merge_t(const AttnParams& p, cudaStream_t stream) {
    merge_kernel<D, G><<<p.B * p.Hkv, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

#define PKV_DISPATCH(D_, G_, ...)                                           \
    switch ((D_) * 16 + (G_)) {                                             \
        case 64 * 16 + 1: { constexpr int kD = 64, kG = 1; __VA_ARGS__; }   \
        case 64 * 16 + 2: { constexpr int kD = 64, kG = 2; __VA_ARGS__; }   \
        case 64 * 16 + 4: { constexpr int kD = 64, kG = 4; __VA_ARGS__; }   \
        case 64 * 16 + 8: { constexpr int kD = 64, kG = 8; __VA_ARGS__; }   \
        case 128 * 16 + 1: { constexpr int kD = 128, kG = 1; __VA_ARGS__; } \
        case 128 * 16 + 2: { constexpr int kD = 128, kG = 2; __VA_ARGS__; } \
        case 128 * 16 + 4: { constexpr int kD = 128, kG = 4; __VA_ARGS__; } \
        case 128 * 16 + 8: { constexpr int kD = 128, kG = 8; __VA_ARGS__; } \
        default: break;                                                     \
    }

// Self-test of the bounded wait: one thread waits on an mbarrier phase that
// nothing completes, through the same wait the pipeline uses, with a short
// limit; the wait must give up, flag PKV_DEV_TIMEOUT and raise the abort flag.
__global__ void wait_selftest_kernel(uint32_t* status, uint64_t limit_ns, int* result) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
    const bool ok = mbar_wait_slow(&bar, 0, status, &abort_flag, limit_ns);   // phase 0 never completes
    const bool again = mbar_wait_slow(&bar, 0, status, &abort_flag, limit_ns);  // after an abort: at once
    result[0] = ok ? 1 : 0;
    result[1] = abort_flag;
    result[2] = again ? 1 : 0;
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, int* result, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns, result);
    return cudaGetLastError();
}

bool shape_supported(int D, int G) {
    PKV_DISPATCH(D, G, (void)kD; (void)kG; return true);
    return false;
}

int attention_ctas_per_sm(int D, int G, bool mma) {
    PKV_DISPATCH(D, G, return mma ? ctas_per_sm_t<kD, kG, true>() : ctas_per_sm_t<kD, kG, false>());
    return 0;
}

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                             cudaStream_t stream, bool cooperative) {
    const int G = p.Hq / p.Hkv;
    PKV_DISPATCH(p.D, G,
                 return p.use_mma ? launch_attention_t<kD, kG, true>(p, kmap, vmap, grid, stream, cooperative)
                                  : launch_attention_t<kD, kG, false>(p, kmap, vmap, grid, stream, cooperative));
    return cudaErrorInvalidValue;
}

cudaError_t launch_resident(const ResidentParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                            cudaStream_t stream) {
    const int G = p.attn.Hq / p.attn.Hkv;
    PKV_DISPATCH(p.attn.D, G,
                 return p.attn.use_mma ? launch_resident_t<kD, kG, true>(p, kmap, vmap, grid, stream)
                                       : launch_resident_t<kD, kG, false>(p, kmap, vmap, grid, stream));
    return cudaErrorInvalidValue;
}

int resident_ctas_per_sm(int D, int G, bool mma) {
    PKV_DISPATCH(D, G, return mma ? resident_ctas_per_sm_t<kD, kG, true>() : resident_ctas_per_sm_t<kD, kG, false>());
    return 0;
}

cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream) {
    const int G = p.Hq / p.Hkv;
    PKV_DISPATCH(p.D, G, return (launch_merge_t<kD, kG>(p, stream)));
    return cudaErrorInvalidValue;
}

}  // namespace pkv

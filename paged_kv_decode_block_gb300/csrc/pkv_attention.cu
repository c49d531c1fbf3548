// pkv_attention.cu -- paged GQA decode attention kernels for GB300 (sm_103a).
//
// Method: "PersistentKV: Page-Aware Decode Scheduling for Long-Context LLM
// Serving on Commodity GPUs" (gist.science summary), Technical Summary,
// Methodology section 1 "Native Block-Table Decode Engine":
//   * one pass over a KV head serves its whole group of G = Hq/Hkv query heads;
//   * K and V are read in place through the block table ("Layout");
//   * a split computes the partial online-softmax state of a disjoint page
//     range and a merge step combines the states exactly ("Sequence Splitting");
//   * split ranges follow the row's true length; an empty split writes the
//     neutral state and reads no KV ("Row-Local Bounds");
//   * tiles come from a compact queue of non-empty (row, KV head, split)
//     intervals ("Compact Workqueue").
// The persistent route drains that queue with an atomic counter, like the
// worker of "GPUOS" (arXiv 2604.17861, section 4.1 "Persistent Kernel
// Executor"), with the grid sized to the SM count as in "WPK persistent kernel"
// (dotwave.ai, "What a persistent kernel is").
//
// GB300 design.  Decode attention reads every KV byte once and does about two
// fp32 FMAs per byte (G = 4), far below the tensor-core balance, so the kernel
// is built for HBM bandwidth on CUDA cores:
//   * one CTA per tile: 4 consumer warps + 1 producer warp;
//   * the producer resolves the block table (32 entries per coalesced load,
//     prefetched one batch ahead) and streams 16-token blocks of K and V into a
//     ring of shared-memory stages with TMA (cp.async.bulk.tensor, L2
//     evict-first), completion tracked by mbarriers;
//   * each consumer warp owns every 4th block and keeps its own online-softmax
//     state (running max m, sum l, fp32 accumulator), so the loop has no
//     CTA-wide barrier; the four states are merged with the same exact LSE rule
//     at the end of the tile;
//   * inside a warp, D/8 lanes cover one 16-byte slice each of a K row; the G
//     partial dot products are summed with a transposing butterfly (each
//     exchange halves the values a lane holds), so a row costs log2(D/8)
//     shuffles per lane instead of G * log2(D/8);
//   * scores are kept in the log2 domain (q pre-scaled by log2(e)/sqrt(D));
//     exp2f is CUDA's own function; everything accumulates in fp32.
// Every wait on an mbarrier is bounded (kWaitLimitNs): on expiry the kernel
// sets PKV_DEV_TIMEOUT in the status word, poisons the tile and carries on.
// Bad page ids set PKV_DEV_PAGE_OOB and poison the tile; no access is made
// through them.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 8;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr unsigned kFull = 0xffffffffu;

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
                                            volatile int* abort) {
    if (abort && *abort) return false;
    const uint64_t start = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - start > kWaitLimitNs) {
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

__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
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
    static constexpr int L = D / 8;                 // lanes per K/V row (16 B each)
    static constexpr int R = 32 / L;                // rows per warp step
    static constexpr int kSteps = kBlockRows / R;   // warp steps per 16-row block
    static constexpr int HG = L / G;                // lanes holding the same head
    static constexpr int kStageElems = kBlockRows * D;
    static constexpr uint32_t kStageBytes = 2u * kStageElems * 2u;  // K + V
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G >= 1 && G <= L, "group size");
};

template <int D, int G>
struct __align__(128) Smem {
    uint16_t k[kStages][kBlockRows * D];
    uint16_t v[kStages][kBlockRows * D];
    float p[kConsumerWarps][kBlockRows * G];   // softmax weights of the block being reduced
    float acc[kConsumerWarps][G * D];          // per-warp states for the end-of-tile merge
    float m[kConsumerWarps][G];
    float l[kConsumerWarps][G];
    int poisoned[kConsumerWarps];
    int bad[kStages];
    uint32_t issued[kStages];   // 1 + use index of the last TMA issued into each stage
    int abort;                  // a wait of this CTA ran out: stop waiting, drain, finish
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int tile_slot[2];
};

struct TileWork {
    int b, kvh;
    int t0, t1;        // token range [t0, t1) of row b (clipped to N_b)
    int slot;          // workspace slot (split tiles)
    int finalize;      // 1: write out/lse directly
    int poisoned;      // plan and device lengths disagree
};

// ------------------------------------------------------------------ tile body

template <int D, int G>
__device__ __forceinline__ void consume_block(const uint16_t* __restrict__ ks, const uint16_t* __restrict__ vs,
                                              float* __restrict__ ps, int valid, int lane,
                                              const float (&qf)[G][8], float (&m)[G], float (&l)[G],
                                              float& m_mine, float (&acc)[G][8]) {
    using C = Cfg<D, G>;
    const int sub = lane % C::L;
    const int rg = lane / C::L;
    const int my_g = sub / C::HG;

    float sc[C::kSteps];
#pragma unroll
    for (int st = 0; st < C::kSteps; ++st) {
        const int row = st * C::R + rg;
        const uint4 raw = *reinterpret_cast<const uint4*>(ks + row * D + sub * 8);
        float kf[8];
        unpack_bf16x8(raw, kf);
        float dot[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float a = qf[g][0] * kf[0];
#pragma unroll
            for (int e = 1; e < 8; ++e) a = fmaf(qf[g][e], kf[e], a);
            dot[g] = a;
        }
        const float s = Butterfly<C::L / 2, G>::run(dot, lane);
        sc[st] = row < valid ? s : -INFINITY;
    }

    // block maximum of my head, then the new running maximum of every head
    float bm = sc[0];
#pragma unroll
    for (int st = 1; st < C::kSteps; ++st) bm = fmaxf(bm, sc[st]);
#pragma unroll
    for (int mask = C::L; mask < 32; mask <<= 1) bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, mask));
    float alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float bmg = __shfl_sync(kFull, bm, g * C::HG);
        const float mn = fmaxf(m[g], bmg);
        alpha[g] = exp2f(m[g] - mn);   // m = -inf on the first block: alpha = 0
        m[g] = mn;
    }
    m_mine = fmaxf(m_mine, bm);

    float pr[C::kSteps];
    float psum = 0.f;
#pragma unroll
    for (int st = 0; st < C::kSteps; ++st) {
        pr[st] = exp2f(sc[st] - m_mine);   // masked rows: exp2(-inf) = 0
        psum += pr[st];
    }
#pragma unroll
    for (int mask = C::L; mask < 32; mask <<= 1) psum += __shfl_xor_sync(kFull, psum, mask);
#pragma unroll
    for (int g = 0; g < G; ++g) {
        l[g] = l[g] * alpha[g] + __shfl_sync(kFull, psum, g * C::HG);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] *= alpha[g];
    }

    // publish p[row][g] for the whole warp, then accumulate p * V
    if (sub % C::HG == 0) {
#pragma unroll
        for (int st = 0; st < C::kSteps; ++st) ps[(st * C::R + rg) * G + my_g] = pr[st];
    }
    __syncwarp();
#pragma unroll
    for (int st = 0; st < C::kSteps; ++st) {
        const int row = st * C::R + rg;
        if (row < valid) {   // rows past N_b may hold stale, even non-finite, data
            const uint4 raw = *reinterpret_cast<const uint4*>(vs + row * D + sub * 8);
            float vf[8];
            unpack_bf16x8(raw, vf);
            float pv[G];
#pragma unroll
            for (int g = 0; g < G; ++g) pv[g] = ps[row * G + g];
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(pv[g], vf[e], acc[g][e]);
        }
    }
    __syncwarp();
}

// Write the neutral state (out = 0, lse = -inf) for every query head of row b.
__device__ void write_neutral_row(const AttnParams& p, int b, int tid, int nthreads) {
    for (int i = tid; i < p.Hq * p.D; i += nthreads) p.out[static_cast<size_t>(b) * p.Hq * p.D + i] = 0.f;
    for (int i = tid; i < p.Hq; i += nthreads) p.lse[static_cast<size_t>(b) * p.Hq + i] = -INFINITY;
}

// Exact LSE merge of the `ns` partial states of (b, kvh) into out / lse.
// Partials come from other CTAs, so they are read through L2 (ld.cg).
template <int D, int G>
__device__ void merge_unit(const AttnParams& p, int b, int kvh, int ns, int tid, int nthreads) {
    const size_t base = static_cast<size_t>(p.row_start[b]) + static_cast<size_t>(kvh) * ns;
    for (int idx = tid; idx < G * D; idx += nthreads) {
        const int g = idx / D, d = idx % D;
        const int h = kvh * G + g;
        float M = -INFINITY;
        bool nan = false;
        for (int s = 0; s < ns; ++s) {
            const float ls = __ldcg(p.ws_lse + (base + s) * G + g);
            nan |= isnan(ls);
            M = fmaxf(M, ls);
        }
        float o = 0.f, lse2 = -INFINITY;
        if (M != -INFINITY) {
            float wsum = 0.f, acc = 0.f;
            for (int s = 0; s < ns; ++s) {
                const float ls = __ldcg(p.ws_lse + (base + s) * G + g);
                const float w = exp2f(ls - M);   // neutral split: exp2(-inf) = 0
                wsum += w;
                acc = fmaf(w, __ldcg(p.ws_o + ((base + s) * G + g) * D + d), acc);
            }
            o = acc / wsum;
            lse2 = M + log2f(wsum);
        }
        if (nan) o = lse2 = NAN;
        p.out[(static_cast<size_t>(b) * p.Hq + h) * D + d] = o;
        if (d == 0) p.lse[static_cast<size_t>(b) * p.Hq + h] = lse2 * 0.69314718055994530942f;
    }
}

// One tile: producer warp streams blocks, consumer warps reduce them, then the
// four warp states are merged and written (to out/lse or to the workspace).
// `pipe` counts blocks this CTA has streamed so far (stage/phase bookkeeping
// continues across the tiles of a persistent CTA).
template <int D, int G>
__device__ void run_tile(Smem<D, G>& sm, const AttnParams& p, const TileWork& tw, uint32_t pipe,
                         const CUtensorMap* kmap, const CUtensorMap* vmap) {
    using C = Cfg<D, G>;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int ntok = tw.t1 > tw.t0 ? tw.t1 - tw.t0 : 0;
    const int nblk = (ntok + kBlockRows - 1) / kBlockRows;
    uint32_t* status = &p.ctr->status;

    if (warp == kConsumerWarps) {
        // ---------------- producer
        if (nblk == 0) return;
        const int ps = p.page_size;
        const int first_page = tw.t0 / ps;
        const int last_page = (tw.t1 + ps - 1) / ps;   // exclusive
        const int32_t* bt_row = p.block_table + static_cast<size_t>(tw.b) * p.max_pages;
        const uint64_t policy = l2_evict_first_policy();
        int j = 0;   // block index within the tile
        int next_id = first_page + lane < last_page ? __ldg(bt_row + first_page + lane) : 0;
        for (int pg0 = first_page; pg0 < last_page; pg0 += 32) {
            const int ids = next_id;
            const int pg_next = pg0 + 32 + lane;
            next_id = pg_next < last_page ? __ldg(bt_row + pg_next) : 0;
            const int n_here = min(32, last_page - pg0);
            for (int i = 0; i < n_here; ++i) {
                const int page = __shfl_sync(kFull, ids, i);
                const int page_tok0 = (pg0 + i) * ps;
                const int lo = max(page_tok0, tw.t0);
                const int hi = min(page_tok0 + ps, tw.t1);
                for (int tok = lo; tok < hi; tok += kBlockRows, ++j) {
                    if (lane == 0) {
                        const uint32_t it = pipe + j;
                        const int s = it % kStages;
                        const uint32_t use = it / kStages;
                        bool go = !sm.abort;
                        if (go && use > 0) go = mbar_wait(&sm.empty[s], (use - 1) & 1u, status, &sm.abort);
                        const bool page_ok = page >= 0 && page < p.num_pages;
                        if (!page_ok) atomicOr(status, static_cast<uint32_t>(PKV_DEV_PAGE_OOB));
                        if (!go || !page_ok) {
                            sm.bad[s] = 1;
                            mbar_arrive(&sm.full[s]);
                        } else {
                            sm.bad[s] = 0;
                            sm.issued[s] = use + 1;
                            mbar_arrive_expect_tx(&sm.full[s], C::kStageBytes);
                            const int row = page * ps + (tok - page_tok0);
                            tma_load_3d(sm.k[s], kmap, 0, tw.kvh, row, &sm.full[s], policy);
                            tma_load_3d(sm.v[s], vmap, 0, tw.kvh, row, &sm.full[s], policy);
                        }
                    }
                }
            }
        }
        return;
    }

    // ---------------- consumers
    const int sub = lane % C::L;
    float qf[G][8];
    {
        const uint16_t* qrow = p.q + (static_cast<size_t>(tw.b) * p.Hq + tw.kvh * G) * D + sub * 8;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow + g * D));
            unpack_bf16x8(raw, qf[g]);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[g][e] *= p.scale_log2;
        }
    }
    float m[G], l[G], acc[G][8];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
    }
    float m_mine = -INFINITY;
    int poisoned = tw.poisoned;

    for (int j = warp; j < nblk; j += kConsumerWarps) {
        const uint32_t it = pipe + j;
        const int s = it % kStages;
        const bool ok = mbar_wait(&sm.full[s], (it / kStages) & 1u, status, &sm.abort);
        if (!ok || sm.bad[s]) {
            poisoned = 1;
        } else {
            const int valid = min(kBlockRows, ntok - j * kBlockRows);
            consume_block<D, G>(sm.k[s], sm.v[s], sm.p[warp], valid, lane, qf, m, l, m_mine, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[s]);
    }

    // fold the row groups of the warp, then publish the warp's state
#pragma unroll
    for (int mask = C::L; mask < 32; mask <<= 1)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(kFull, acc[g][e], mask);
    if (lane < C::L) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < 8; ++e) sm.acc[warp][g * D + sub * 8 + e] = acc[g][e];
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            sm.m[warp][g] = m[g];
            sm.l[warp][g] = l[g];
        }
        sm.poisoned[warp] = poisoned;
    }
    named_barrier_sync(1, kConsumerWarps * 32);

    const int tid = threadIdx.x;
    bool any_poison = false;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) any_poison |= sm.poisoned[w] != 0;
    for (int idx = tid; idx < G * D; idx += kConsumerWarps * 32) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.m[w][g]);
        float o = 0.f, lse2 = -INFINITY;
        if (M != -INFINITY) {
            float lsum = 0.f, osum = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) {
                const float sc = exp2f(sm.m[w][g] - M);   // idle warp: m = -inf -> 0
                lsum = fmaf(sm.l[w][g], sc, lsum);
                osum = fmaf(sm.acc[w][g * D + d], sc, osum);
            }
            o = osum / lsum;
            lse2 = M + log2f(lsum);
        }
        if (any_poison) o = lse2 = NAN;
        if (tw.finalize) {
            const int h = tw.kvh * G + g;
            p.out[(static_cast<size_t>(tw.b) * p.Hq + h) * D + d] = o;
            if (d == 0) p.lse[static_cast<size_t>(tw.b) * p.Hq + h] = lse2 * 0.69314718055994530942f;
        } else {
            p.ws_o[(static_cast<size_t>(tw.slot) * G + g) * D + d] = o;
            if (d == 0) p.ws_lse[static_cast<size_t>(tw.slot) * G + g] = lse2;
        }
    }
}

// After an abort, wait (bounded again) for every TMA copy this CTA issued, so
// that none lands in shared memory after the CTA has moved on or exited.
// Called by one thread once the producer has stopped issuing.
template <int D, int G>
__device__ void drain_after_abort(Smem<D, G>& sm, uint32_t* status) {
    for (int s = 0; s < kStages; ++s)
        if (sm.issued[s] > 0) mbar_wait_slow(&sm.full[s], (sm.issued[s] - 1) & 1u, status, nullptr);
}

// Tile of a queue entry, with the plan checked against the device lengths.
__device__ __forceinline__ TileWork tile_from_queue(const AttnParams& p, int t) {
    const pkv_work_item it = p.queue[t];
    TileWork tw;
    tw.b = it.b;
    tw.kvh = it.kvh;
    const int n = p.seq_lens[it.b];
    const int pages = (n + p.page_size - 1) / p.page_size;
    const int splits = p.row_splits[it.b];
    const int want_end = min((it.split + 1) * p.chunk_pages, pages);
    tw.poisoned = (it.page_begin != it.split * p.chunk_pages || it.page_end != want_end) ? 1 : 0;
    if (tw.poisoned && threadIdx.x == 0) atomicOr(&p.ctr->status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
    tw.t0 = it.page_begin * p.page_size;
    tw.t1 = min(it.page_end * p.page_size, n);
    if (tw.poisoned) tw.t1 = tw.t0;   // read nothing through a plan that does not fit
    tw.finalize = splits == 1;
    tw.slot = p.row_start[it.b] + it.kvh * splits + it.split;
    return tw;
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads) attention_kernel(const AttnParams p,
                                                             const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap vmap) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<D, G>& sm = *reinterpret_cast<Smem<D, G>*>(smem_raw);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
            sm.issued[s] = 0;
        }
        sm.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (p.route == kRoutePersistent) {
        // rows with no tokens get no tiles: write their neutral state here
        for (int b = blockIdx.x; b < p.B; b += gridDim.x)
            if (p.row_splits[b] == 0) write_neutral_row(p, b, threadIdx.x, blockDim.x);
        uint32_t pipe = 0;
        while (true) {
            if (threadIdx.x == 0) sm.tile_slot[0] = static_cast<int>(atomicAdd(&p.ctr->next_tile, 1u));
            __syncthreads();
            const int t = sm.tile_slot[0];
            if (t >= p.num_tiles) break;
            const TileWork tw = tile_from_queue(p, t);
            run_tile<D, G>(sm, p, tw, pipe, &kmap, &vmap);
            const int ntok = tw.t1 > tw.t0 ? tw.t1 - tw.t0 : 0;
            pipe += (ntok + kBlockRows - 1) / kBlockRows;
            if (!tw.finalize && p.fused_merge) {
                // last-arriving split of (b, kvh) merges all of them
                __threadfence();
                __syncthreads();
                if (threadIdx.x == 0) {
                    const int u = tw.b * p.Hkv + tw.kvh;
                    const int ns = p.row_splits[tw.b];
                    const uint32_t prev = atomicAdd(&p.arrive[u], 1u);
                    const int last = prev == static_cast<uint32_t>(ns - 1);
                    if (last) p.arrive[u] = 0;   // ready for the next launch
                    sm.tile_slot[1] = last;
                }
                __syncthreads();
                if (sm.tile_slot[1]) {
                    __threadfence();
                    merge_unit<D, G>(p, tw.b, tw.kvh, p.row_splits[tw.b], threadIdx.x, blockDim.x);
                }
            }
            __syncthreads();
        }
        if (threadIdx.x == 0) {
            if (sm.abort) drain_after_abort<D, G>(sm, &p.ctr->status);
            // the last CTA out rewinds the queue for the next launch
            if (atomicAdd(&p.ctr->done_ctas, 1u) == gridDim.x - 1) {
                p.ctr->next_tile = 0;
                p.ctr->done_ctas = 0;
            }
        }
        return;
    }

    TileWork tw;
    if (p.route == kRouteDirect) {
        tw.b = blockIdx.x / p.Hkv;
        tw.kvh = blockIdx.x % p.Hkv;
        tw.t0 = 0;
        tw.t1 = p.seq_lens[tw.b];
        tw.slot = 0;
        tw.finalize = 1;
        tw.poisoned = 0;
        if (tw.t1 > p.max_pages * p.page_size) {   // would read past the table row
            tw.poisoned = 1;
            tw.t1 = 0;
            if (threadIdx.x == 0) atomicOr(&p.ctr->status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
        }
    } else if (p.route == kRouteQueue) {
        tw = tile_from_queue(p, blockIdx.x);
    } else {   // padded grid: (b, kvh, s) from the block index, ranges from the device lengths
        const int per_row = p.Hkv * p.max_splits;
        tw.b = blockIdx.x / per_row;
        tw.kvh = (blockIdx.x % per_row) / p.max_splits;
        const int s = blockIdx.x % p.max_splits;
        const int n = p.seq_lens[tw.b];
        const int pages = (n + p.page_size - 1) / p.page_size;
        tw.poisoned = pages > p.max_splits * p.chunk_pages || n > p.max_pages * p.page_size;
        if (tw.poisoned && threadIdx.x == 0) atomicOr(&p.ctr->status, static_cast<uint32_t>(PKV_DEV_PLAN_MISMATCH));
        const int pb = min(s * p.chunk_pages, pages);
        const int pe = min((s + 1) * p.chunk_pages, pages);
        tw.t0 = pb * p.page_size;
        tw.t1 = tw.poisoned ? tw.t0 : min(pe * p.page_size, n);
        tw.finalize = p.max_splits == 1;
        tw.slot = blockIdx.x;
    }
    run_tile<D, G>(sm, p, tw, 0, &kmap, &vmap);
    __syncthreads();
    if (threadIdx.x == 0 && sm.abort) drain_after_abort<D, G>(sm, &p.ctr->status);
}

template <int D, int G>
__global__ void __launch_bounds__(128) merge_kernel(const AttnParams p) {
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
    merge_unit<D, G>(p, b, kvh, ns, threadIdx.x, blockDim.x);
}

template <int D, int G>
cudaError_t launch_attention_t(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                               cudaStream_t stream) {
    const size_t smem = sizeof(Smem<D, G>);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(attention_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    attention_kernel<D, G><<<grid, kThreads, smem, stream>>>(p, kmap, vmap);
    return cudaGetLastError();
}

template <int D, int G>
int ctas_per_sm_t() {
    const size_t smem = sizeof(Smem<D, G>);
    if (cudaFuncSetAttribute(attention_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attention_kernel<D, G>, kThreads, smem) != cudaSuccess)
        return 0;
    return n;
}

template <int D, int G>
cudaError_t launch_merge_t(const AttnParams& p, cudaStream_t stream) {
    merge_kernel<D, G><<<p.B * p.Hkv, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

#define PKV_DISPATCH(D_, G_, CALL)                                   \
    switch ((D_) * 16 + (G_)) {                                      \
        case 64 * 16 + 1: { constexpr int kD = 64, kG = 1; CALL; }   \
        case 64 * 16 + 2: { constexpr int kD = 64, kG = 2; CALL; }   \
        case 64 * 16 + 4: { constexpr int kD = 64, kG = 4; CALL; }   \
        case 64 * 16 + 8: { constexpr int kD = 64, kG = 8; CALL; }   \
        case 128 * 16 + 1: { constexpr int kD = 128, kG = 1; CALL; } \
        case 128 * 16 + 2: { constexpr int kD = 128, kG = 2; CALL; } \
        case 128 * 16 + 4: { constexpr int kD = 128, kG = 4; CALL; } \
        case 128 * 16 + 8: { constexpr int kD = 128, kG = 8; CALL; } \
        default: break;                                              \
    }

}  // namespace

bool shape_supported(int D, int G) {
    PKV_DISPATCH(D, G, (void)kD; (void)kG; return true);
    return false;
}

int attention_ctas_per_sm(int D, int G) {
    PKV_DISPATCH(D, G, return (ctas_per_sm_t<kD, kG>()));
    return 0;
}

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap, int grid,
                             cudaStream_t stream) {
    const int G = p.Hq / p.Hkv;
    PKV_DISPATCH(p.D, G, return (launch_attention_t<kD, kG>(p, kmap, vmap, grid, stream)));
    return cudaErrorInvalidValue;
}

cudaError_t launch_merge(const AttnParams& p, cudaStream_t stream) {
    const int G = p.Hq / p.Hkv;
    PKV_DISPATCH(p.D, G, return (launch_merge_t<kD, kG>(p, stream)));
    return cudaErrorInvalidValue;
}

}  // namespace pkv

// kvi_shared.cu -- many queries against one shared fact store.
//
// "InferScale: GPU-Native KV Injection for Personalized LLM Serving",
// Section 6.4: concurrent users issue queries against one conversation's
// memory store.  Scoring R queries against the same N x E embedding matrix
// is a dense contraction S = Q E^T, so here it runs on the 5th-generation
// tensor cores instead of R separate scans of the matrix:
//
//   coarse_kernel   (more than 128 queries) one CTA per 128 facts.  A TMA
//                   producer warp (one box per lane) streams the facts' rows
//                   and all queries through a ring of 128-byte swizzled
//                   stages; one thread issues tcgen05.mma (kind::tf32,
//                   M = 128, N = R padded to 16) accumulating in tensor
//                   memory; four warps compute the row norms from the same
//                   stages and, at the end, read the accumulator back
//                   (tcgen05.ld) and write an interval [lo, hi] that provably
//                   holds every exact score (bound below).
//   coarse_split_kernel  (up to 128 queries) the same pipeline with the
//                   queries on M and up to 256 facts on N, each tile's K
//                   range split over a thread-block cluster (below).
//   then, per query (kvi_retrieve.cu): the facts whose hi reaches a lower
//   bound of the k-th lo are collected in id order, rescored exactly (the
//   Dot2 key of the plain path) and ranked by the plain selector, so the
//   result is the exact top-k of the plain path, tie for tie.
//
// Bound.  TF32 keeps 10 mantissa bits of each operand, so each product
// carries a relative error below 2^-9 + 2^-20; the float32 accumulation of E
// products adds at most E * 2^-23 of the running magnitude.  With
// sum_j |q_j e_j| <= |q| |e| (Cauchy-Schwarz) the exact score lies within
// eps = (2^-9 + E 2^-23) |q| |e| of the tensor-core value; the kernel uses
// four times that, plus 2^-100 for flushed subnormals, and rounds lo down
// and hi up.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "kvi_internal.cuh"

namespace kvi {

#ifdef KVI_DEBUG_CHECKS
// Debug builds: the (CTA, K chunk) whose stage the coarse kernels do not
// load (CTA < 0: none), set by kvi_debug_stall_coarse_chunk.
__device__ int g_debug_stall_cta = -1;
__device__ int g_debug_stall_chunk = -1;
#endif

namespace {

constexpr int kTileM = 128;          // facts per CTA (MMA M)
constexpr int kChunk = 32;           // float32 per row per stage: one 128-byte swizzle row
constexpr int kCoarseThreads = 192;  // warp 0 TMA, warp 1 MMA + TMEM, warps 2-5 norms + epilogue
constexpr int kStageBytesA = kTileM * kChunk * 4;
constexpr int kRingBudget = 200 * 1024;
constexpr int kMaxStages = 8;
// Rows per TMA box: a whole 128-fact accumulator tile per box (16 KB), and
// up to 128 query rows per box.  Each tensor copy has a fixed cost in the
// SM's copy unit, so fewer, larger boxes per stage move a stage sooner.
constexpr int kBoxRowsA = 128;
constexpr int kBoxRowsBMax = 128;
constexpr uint64_t kWaitNs = 1000000000ull;

struct CoarseSmemTail {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t pad;
    float qscale[KVI_MAX_SHARED_QUERIES];  // rel * |q_r| per query (see the epilogue)
};

__device__ __forceinline__ uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity)
{
    if (try_wait(bar, parity)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        if (try_wait(bar, parity)) return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > kWaitNs) return false;
    }
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout TMA writes: rows of 128 bytes, 8-row groups 1024 bytes
// apart (stride byte offset), descriptor version 1, layout type 2.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr)
{
    uint64_t d = (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;              // leading byte offset: unused for swizzled K-major
    d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset
    d |= (uint64_t)1 << 46;              // descriptor version
    d |= (uint64_t)2 << 61;              // 128-byte swizzle
    return d;
}

// Instruction descriptor: D float32, A and B tf32, both K-major, M x N.
__device__ __forceinline__ uint32_t tf32_idesc(int m, int n)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Sum of squares of one 128-byte row chunk.  Lane l starts at 16-byte column
// l mod 8: the lanes of a warp read 32 different rows, whose same column
// lies in the same four banks (rows are 128 bytes apart), so reading column
// c in step c would be a 32-way bank conflict; rotated, each step touches
// all eight columns and takes the minimum four shared-memory wavefronts.
__device__ __forceinline__ float sq_row32(const float *row, int rot)
{
    const float4 *r4 = reinterpret_cast<const float4 *>(row);
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < kChunk / 4; ++c) {
        const float4 v = r4[(c + rot) & (kChunk / 4 - 1)];
        acc = fmaf(v.x, v.x, acc);
        acc = fmaf(v.y, v.y, acc);
        acc = fmaf(v.z, v.z, acc);
        acc = fmaf(v.w, v.w, acc);
    }
    return acc;
}

__global__ void __launch_bounds__(kCoarseThreads, 1)
coarse_kernel(const __grid_constant__ CUtensorMap tm_emb, const __grid_constant__ CUtensorMap tm_q,
              const __grid_constant__ CoarseParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned stages: A (facts) then B (queries), then the tail
    uint8_t *base = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = p.stages;
    // MT accumulators of kTileM facts each share every query chunk
    const int MT = p.mt;
    const int stage_a = MT * kStageBytesA;
    const int stage_b = p.Rp * kChunk * 4;
    uint8_t *a_st = base;
    uint8_t *b_st = base + (size_t)S * stage_a;
    CoarseSmemTail &tl = *reinterpret_cast<CoarseSmemTail *>(b_st + (size_t)S * stage_b);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x;
    const int nk = (p.E + kChunk - 1) / kChunk;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&tl.full[s])) : "memory");
            // the MMA commit plus one arrival from each of the four norm warps
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 5;" ::"r"(saddr(&tl.empty[s])) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&tl.mma_done)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tl.tmem_base)),
                     "r"((uint32_t)p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tl.tmem_base;
    pdl_launch_dependents();  // the candidate kernel may be scheduled; it waits for this grid's end
    const int cols_acc = p.tmem_cols / MT;  // tensor-memory columns per accumulator
    bool ok = true;

    if (warp == 0) {
        // the stage is loaded as boxes of kBoxRowsA fact rows and box_q
        // query rows, one box per lane (a single issuing thread caps the
        // copy rate far below the SM's share of HBM bandwidth)
        const uint32_t bytes = (uint32_t)(stage_a + stage_b);
        const int bq = p.box_q;  // query rows per box
        const int na = MT * kTileM / kBoxRowsA, nb = (p.Rp + bq - 1) / bq;
        int issued = 0;  // chunks whose copies went out
        // stage and round of chunk kc, kept as counters (a division by the
        // run-time stage count would sit on every stage's critical path)
        int s = 0, round = 0;
        for (int kc = 0; kc < nk; ++kc) {
            bool go = true;
            if (lane == 0 && round > 0) go = wait_bar(saddr(&tl.empty[s]), (uint32_t)((round - 1) & 1));
            if (!__shfl_sync(0xffffffffu, go ? 1 : 0, 0)) {
                if (lane == 0) record_status(p.status, KVI_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const uint32_t fb = saddr(&tl.full[s]);
#ifdef KVI_DEBUG_CHECKS
            // no expect-tx and no copy for this chunk: the waits on its
            // stage run out
            const bool stall = (int)blockIdx.x == g_debug_stall_cta && kc == g_debug_stall_chunk;
#else
            constexpr bool stall = false;
#endif
            if (lane == 0 && !stall) {
                if (round > 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(bytes) : "memory");
            }
            __syncwarp();
            for (int j = lane; j < (stall ? 0 : na + nb); j += 32) {
                if (j < na)
                    tma_2d(saddr(a_st + (size_t)s * stage_a + (size_t)j * kBoxRowsA * 128), &tm_emb,
                           kc * kChunk, tile * MT * kTileM + j * kBoxRowsA, fb);
                else
                    tma_2d(saddr(b_st + (size_t)s * stage_b + (size_t)(j - na) * bq * 128), &tm_q,
                           kc * kChunk, (j - na) * bq, fb);
            }
            issued = kc + 1;
            if (++s == S) {
                s = 0;
                ++round;
            }
        }
        // no copy may still be writing into shared memory when the CTA
        // ends: wait (bounded) for the last chunk issued into every stage
        if (lane < S && lane < issued) {
            const int r = (issued - 1 - lane) / S;  // round of stage `lane`'s last chunk
            if (!wait_bar(saddr(&tl.full[lane]), (uint32_t)(r & 1))) record_status(p.status, KVI_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tf32_idesc(kTileM, p.Rp);
            int s = 0;
            uint32_t ph = 0;  // phase parity of stage s's full barrier
            for (int kc = 0; kc < nk; ++kc) {
                if (!wait_bar(saddr(&tl.full[s]), ph)) {
                    record_status(p.status, KVI_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a0 = saddr(a_st + (size_t)s * stage_a);
                const uint32_t b0 = saddr(b_st + (size_t)s * stage_b);
#pragma unroll
                for (int kk = 0; kk < kChunk / 8; ++kk) {  // K = 8 tf32 (32 bytes) per MMA
                    const uint64_t bd = sw128_desc(b0 + 32u * kk);
                    const uint32_t acc = (kc > 0 || kk > 0) ? 1u : 0u;
                    // accumulator m: fact rows 128 m .. 128 m + 127 of the
                    // stage (16 KB further on), columns m * cols_acc on
                    for (int m = 0; m < MT; ++m) {
                        const uint64_t ad = sw128_desc(a0 + (uint32_t)(m * kStageBytesA) + 32u * kk);
                        asm volatile(
                            "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(
                                tmem + (uint32_t)(m * cols_acc)),
                            "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
                            : "memory");
                    }
                }
                // the stage is free once these MMAs have read it
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 saddr(&tl.empty[s]))
                             : "memory");
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            // committed whatever ended the loop, so that the MMAs issued
            // are known complete before tensor memory is released; after a
            // timeout the intervals are not valid (the status says so)
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             saddr(&tl.mma_done))
                         : "memory");
            if (!wait_bar(saddr(&tl.mma_done), 0)) record_status(p.status, KVI_ERR_TIMEOUT);
        }
    } else {
        // warps 2-5: thread L owns tensor-memory lane L = fact row L of the
        // tile (a warp reaches the 32 lanes of its own subpartition, warp % 4)
        const int q = warp & 3;
        const int L = 32 * q + lane;
        float en2[2] = {0.f, 0.f}, qa = 0.f, qb = 0.f;  // en2[m]: fact row 128 m + L
        int s = 0;
        uint32_t ph = 0;
        for (int kc = 0; kc < nk; ++kc) {
            const bool got = wait_bar(saddr(&tl.full[s]), ph);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) record_status(p.status, KVI_ERR_TIMEOUT);
                ok = false;
                break;
            }
            // a row's 128 bytes stay within its own 128-byte span under the
            // swizzle (only their 16-byte chunks are permuted), so a sum of
            // squares reads them in place
            en2[0] += sq_row32(reinterpret_cast<const float *>(a_st + (size_t)s * stage_a + L * 128), lane);
            if (MT == 2)
                en2[1] += sq_row32(
                    reinterpret_cast<const float *>(a_st + (size_t)s * stage_a + kStageBytesA + L * 128), lane);
            if (L < p.Rp)
                qa += sq_row32(reinterpret_cast<const float *>(b_st + (size_t)s * stage_b + L * 128), lane);
            if (L + 128 < p.Rp)
                qb += sq_row32(reinterpret_cast<const float *>(b_st + (size_t)s * stage_b + (L + 128) * 128), lane);
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&tl.empty[s])) : "memory");
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        // the bound's per-query factor, once per query row instead of once
        // per (fact, query) in the epilogue
        const float rel = (0.001953125f + (float)p.E * 1.1920929e-7f) * 4.0f;  // 4 (2^-9 + E 2^-23)
        if (L < p.Rp) tl.qscale[L] = rel * sqrtf(qa);
        if (L + 128 < p.Rp) tl.qscale[L + 128] = rel * sqrtf(qb);
        asm volatile("bar.sync 1, 128;" ::: "memory");
        const bool done = ok && wait_bar(saddr(&tl.mma_done), 0);
        if (__all_sync(0xffffffffu, done)) {
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            for (int m = 0; m < MT; ++m) {
            const int64_t fact = ((int64_t)tile * MT + m) * kTileM + L;
            const float en = sqrtf(m == 0 ? en2[0] : en2[1]);
            for (int c0 = 0; c0 < p.Rp; c0 += 16) {
                uint32_t v[16];
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
                    "%15}, [%16];"
                    : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
                      "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
                      "=r"(v[14]), "=r"(v[15])
                    : "r"(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(m * cols_acc + c0)));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (fact < p.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int r = c0 + j;
                        if (r < p.R) {
                            const float c = __uint_as_float(v[j]);
                            const float eps = __fmaf_ru(tl.qscale[r], en * 1.0001f, 7.9e-31f);
                            p.lo[(int64_t)r * p.stride + fact] = __fsub_rd(c, eps);
                            p.hi[(int64_t)r * p.stride + fact] = __fadd_ru(c, eps);
                        }
                    }
                }
            }
            }
        } else if (lane == 0) {
            record_status(p.status, KVI_ERR_TIMEOUT);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)p.tmem_cols)
                     : "memory");
    }
}

// ------------------------------------------------------- split form, R <= 128
//
// Each tcgen05.mma of kind::tf32 costs the issuing SM about the same time
// whatever its N (measured: 4 MMAs of K = 8 take ~670 cycles at N = 64 and
// at N = 256), so a CTA's run time is set by the E / 8 instructions of its
// K loop, not by its bytes.  With at most 128 queries the split form puts
// the queries on M (one 128-row accumulator) and up to 256 facts on N, which
// needs 2 to 4 times fewer instructions than facts on M; and it splits each
// tile's K range over a cluster of `split` CTAs, so that each runs only
// E / (8 split) of them.  After the loops the tile's 32-column groups are
// shared out round robin: each CTA sends its partial accumulator of the
// groups the others finalize, and its partial squared norms, into their
// (idle) rings through distributed shared memory; each then adds the parts
// of its own groups and writes their intervals with tensor stores.  The
// partial sums are one more summation order of the same E products, so the
// float32 accumulation term of the bound is unchanged.

constexpr int kQTile = 128;               // MMA M: query rows (at most 128 of them queries)
constexpr int kSlotQ = kQTile * kChunk * 4;
constexpr int kMaxF = 256;                // MMA N: facts per tile
constexpr int kMaxSplit = 4;
// warp 0 TMA, warp 1 MMA + TMEM, warps 2-7 norms; after the K loop all eight
// warps take part, two per tensor-memory subpartition
constexpr int kSplitThreads = 256;

struct SplitSmemTail {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t mma_done;
    uint32_t tmem_base;
    uint32_t acc_ok;       // the MMA thread saw every MMA complete
    float en2[kMaxF];      // this CTA's squared fact norms over its K range
    float qa2[kQTile];     // and squared query norms
    float fnorm[kMaxF];    // |e| per fact of the tile (all K)
    float qscale[kQTile];  // rel * |q| per query (all K)
};

// Fact rows per tensor copy: no copy exceeds 128 rows of 128 bytes (F is a
// multiple of 32, so F / 2 is a multiple of 16)
__host__ __device__ constexpr int split_fact_box(int F) { return F > 128 ? F / 2 : F; }

// The tile's 32-column groups are finalized round robin: group g by the
// cluster's CTA g % split.  Each CTA receives, from each of the other
// split - 1 CTAs, a part in its (idle) ring: that CTA's partial accumulator
// of the groups this one finalizes, column by column ([groups][32][Rp]
// floats), then its squared norms ([256] facts, [128] queries).
__host__ __device__ constexpr int split_groups_owned(int F, int P) { return (F / 32 + P - 1) / P; }
__host__ __device__ constexpr size_t split_part_bytes(int Rp, int F, int P)
{
    return (((size_t)split_groups_owned(F, P) * 32 * Rp + kMaxF + kQTile) * 4 + 15) & ~(size_t)15;
}
// After the parts, each warp's output staging: a lo and a hi box of
// 32 x 32 floats, 1024-byte aligned for the 128-byte swizzle
constexpr int kOutBoxBytes = 32 * 32 * 4;
constexpr size_t kOutStageBytes = 8 * 2 * kOutBoxBytes;
__host__ __device__ constexpr size_t split_out_offset(int P, size_t part)
{
    return ((size_t)(P - 1) * part + 1023) & ~(size_t)1023;
}

// Shared-memory accesses by 32-bit shared address (ld/st.shared): the
// compiler cannot take them for global accesses that they might alias.
__device__ __forceinline__ float lds_f32(uint32_t a)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ void sts_v4(uint32_t a, float x, float y, float z, float w)
{
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(x), "f"(y), "f"(z), "f"(w) : "memory");
}

// Tensor store of one box from shared memory (bulk group of this thread)
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

// 32 consecutive tensor-memory columns of this warp's 32 lanes: lane t gets
// row t, columns c .. c + 31 in v[0..31]
__device__ __forceinline__ void tmem_ld32(uint32_t addr, uint32_t (&v)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_addr(uint32_t a, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t a, float x)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(a), "f"(x) : "memory");
}

// Every thread of every CTA of the cluster (the release/acquire pair also
// orders the distributed shared-memory writes before the reads).
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release;\nbarrier.cluster.wait.acquire;" ::: "memory");
}

__global__ void __launch_bounds__(kSplitThreads, 1)
coarse_split_kernel(const __grid_constant__ CUtensorMap tm_emb, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_lo, const __grid_constant__ CUtensorMap tm_hi,
                    const __grid_constant__ CoarseParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int S = p.stages, F = p.F, P = p.split;
    const int stage_f = F * kChunk * 4;
    uint8_t *q_st = base;                       // S slots of 128 query rows
    uint8_t *f_st = base + (size_t)S * kSlotQ;  // S slots of F fact rows
    SplitSmemTail &tl = *reinterpret_cast<SplitSmemTail *>(f_st + (size_t)S * stage_f);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tile = blockIdx.x / P, rank = blockIdx.x % P;  // rank: this CTA's place in its cluster
    const int64_t f0 = (int64_t)tile * F;
    const int nk = (p.E + kChunk - 1) / kChunk;
    const int k0 = rank * nk / P, k1 = (rank + 1) * nk / P;  // this CTA's K chunks

    if (tid == 0) {
        // the copy descriptors are fetched while the barriers are set up
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_emb)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
        for (int s = 0; s < S; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&tl.full[s])) : "memory");
            // the MMA commit plus one arrival from each of the six norm warps
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 7;" ::"r"(saddr(&tl.empty[s])) : "memory");
        }
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(saddr(&tl.mma_done)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    // rows that no norm thread owns (facts past F, queries past Rp) stay 0
    tl.en2[tid] = 0.f;
    if (tid < kQTile) tl.qa2[tid] = 0.f;
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(&tl.tmem_base)),
                     "r"((uint32_t)p.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tl.tmem_base;
    pdl_launch_dependents();  // the candidate kernel may be scheduled; it waits for this grid's end
    bool ok = true;
    const int L = 32 * (warp & 3) + lane;  // tensor-memory lane of this thread = query row

    if (warp == 0) {
        // per chunk: the query rows as boxes of box_q rows (they tile Rp
        // exactly) and the tile's F fact rows as one or two boxes, one box
        // per lane
        const uint32_t bytes = (uint32_t)((p.Rp + F) * kChunk * 4);
        const int bq = p.box_q, nb = p.Rp / bq;
        // facts in boxes of at most 128 rows (16 KB): one, or two halves
        const int bf = split_fact_box(F), nfb = F / bf;
        int issued = 0, s = 0, round = 0;
        for (int kc = k0; kc < k1; ++kc) {
            bool go = true;
            if (lane == 0 && round > 0) go = wait_bar(saddr(&tl.empty[s]), (uint32_t)((round - 1) & 1));
            if (!__shfl_sync(0xffffffffu, go ? 1 : 0, 0)) {
                if (lane == 0) record_status(p.status, KVI_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const uint32_t fb = saddr(&tl.full[s]);
#ifdef KVI_DEBUG_CHECKS
            // no expect-tx and no copy for this chunk: the waits on its
            // stage run out
            const bool stall = (int)blockIdx.x == g_debug_stall_cta && kc == g_debug_stall_chunk;
#else
            constexpr bool stall = false;
#endif
            if (lane == 0 && !stall) {
                if (round > 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(bytes) : "memory");
            }
            __syncwarp();
            for (int j = lane; j < (stall ? 0 : nb + nfb); j += 32) {
                if (j < nb)
                    tma_2d(saddr(q_st + (size_t)s * kSlotQ + (size_t)j * bq * 128), &tm_q, kc * kChunk, j * bq, fb);
                else
                    tma_2d(saddr(f_st + (size_t)s * stage_f + (size_t)(j - nb) * bf * 128), &tm_emb, kc * kChunk,
                           (int)f0 + (j - nb) * bf, fb);
            }
            ++issued;
            if (++s == S) {
                s = 0;
                ++round;
            }
        }
        // no copy may still be writing into shared memory when the ring is
        // reused or the CTA ends: wait (bounded) for each stage's last chunk
        if (lane < S && lane < issued) {
            const int r = (issued - 1 - lane) / S;
            if (!wait_bar(saddr(&tl.full[lane]), (uint32_t)(r & 1))) record_status(p.status, KVI_ERR_TIMEOUT);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tf32_idesc(kQTile, F);
            int s = 0;
            uint32_t ph = 0;
            for (int kc = k0; kc < k1; ++kc) {
                if (!wait_bar(saddr(&tl.full[s]), ph)) {
                    record_status(p.status, KVI_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
                const uint32_t a0 = saddr(q_st + (size_t)s * kSlotQ);
                const uint32_t b0 = saddr(f_st + (size_t)s * stage_f);
#pragma unroll
                for (int kk = 0; kk < kChunk / 8; ++kk) {  // K = 8 tf32 (32 bytes) per MMA
                    const uint64_t ad = sw128_desc(a0 + 32u * kk);
                    const uint64_t bd = sw128_desc(b0 + 32u * kk);
                    const uint32_t acc = (kc > k0 || kk > 0) ? 1u : 0u;
                    asm volatile(
                        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem),
                        "l"(ad), "l"(bd), "r"(idesc), "r"(acc)
                        : "memory");
                }
                asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                                 saddr(&tl.empty[s]))
                             : "memory");
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             saddr(&tl.mma_done))
                         : "memory");
            const bool done = ok && wait_bar(saddr(&tl.mma_done), 0);
            if (!done) record_status(p.status, KVI_ERR_TIMEOUT);
            tl.acc_ok = done ? 1u : 0u;
        }
    } else {
        // warps 2-7 (192 threads): squared norms over this CTA's chunks of
        // the F fact rows and then the Rp query rows of each stage; thread t
        // owns rows t and t + 192 of that list (consecutive rows per warp)
        const int t = tid - 64;
        const int nrows = F + p.Rp;
        float a0 = 0.f, a1 = 0.f;
        int s = 0;
        uint32_t ph = 0;
        for (int kc = k0; kc < k1; ++kc) {
            const bool got = wait_bar(saddr(&tl.full[s]), ph);
            if (!__all_sync(0xffffffffu, got)) {
                if (lane == 0) record_status(p.status, KVI_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const uint8_t *fs = f_st + (size_t)s * stage_f;
            const uint8_t *qs = q_st + (size_t)s * kSlotQ;
            if (t < nrows)
                a0 += sq_row32(reinterpret_cast<const float *>(t < F ? fs + t * 128 : qs + (t - F) * 128), lane);
            if (t + 192 < nrows)
                a1 += sq_row32(
                    reinterpret_cast<const float *>(t + 192 < F ? fs + (t + 192) * 128 : qs + (t + 192 - F) * 128),
                    lane);
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(&tl.empty[s])) : "memory");
            if (++s == S) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (t < nrows) (t < F ? tl.en2[t] : tl.qa2[t - F]) = a0;
        if (t + 192 < nrows) (t + 192 < F ? tl.en2[t + 192] : tl.qa2[t + 192 - F]) = a1;
    }

    const int G = F / 32;                      // 32-column groups of the tile
    const int gown = split_groups_owned(F, P);  // most groups one CTA finalizes
    const size_t part = split_part_bytes(p.Rp, F, P);
    const uint32_t ring = saddr(base);
    // from here every warp takes part: its tensor-memory lanes hold query
    // rows 32 (warp % 4) .. + 31, and the two warps of a subpartition take
    // alternate column groups (half = warp / 4)
    const int row0 = 32 * (warp & 3), half = warp >> 2;
    const bool rows_here = row0 < p.R;
    const bool norm_warp = warp >= 2 && warp < 6;
    const uint32_t tm_rows = tmem + ((uint32_t)row0 << 16);
    if (P > 1)
        cluster_sync_all();  // every CTA's MMAs are done and every ring is idle
    else
        __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // (after a timeout the status word is set and no interval is written)
    const bool acc_ok = tl.acc_ok != 0;
    if (P > 1) {
        // partials of the groups that other CTAs finalize, into their
        // rings; lanes are consecutive rows, so each store is 128 bytes
        if (rows_here && acc_ok) {
            int i = 0;  // index among the groups that others finalize
            for (int g = 0; g < G; ++g) {
                const int o = g % P;
                if (o == rank) continue;
                if ((i++ & 1) != half) continue;
                const int sidx = rank < o ? rank : rank - 1;  // this CTA among o's senders
                const uint32_t dst =
                    cluster_addr(ring, (uint32_t)o) + (uint32_t)(sidx * part) + (uint32_t)((g / P) * 32 * p.Rp * 4);
                __syncwarp();
                uint32_t v[32];
                tmem_ld32(tm_rows + (uint32_t)(32 * g), v);
                if (L < p.R) {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        st_cluster_f32(dst + (uint32_t)((j * p.Rp + L) * 4), __uint_as_float(v[j]));
                }
            }
        }
        // squared norms over this CTA's K range, to every other CTA
        if (norm_warp) {
            for (int o = 0; o < P; ++o) {
                if (o == rank) continue;
                const int sidx = rank < o ? rank : rank - 1;
                const uint32_t nrm =
                    cluster_addr(ring, (uint32_t)o) + (uint32_t)(sidx * part) + (uint32_t)(gown * 32 * p.Rp * 4);
                st_cluster_f32(nrm + 4u * L, tl.en2[L]);
                st_cluster_f32(nrm + 4u * (L + 128), tl.en2[L + 128]);
                st_cluster_f32(nrm + 4u * (kMaxF + L), tl.qa2[L]);
            }
        }
        cluster_sync_all();  // the parts are in place
    }
    if (norm_warp) {
        // totals over the cluster's K ranges: |e| per fact, rel |q| per query
        const float rel = (0.001953125f + (float)p.E * 1.1920929e-7f) * 4.0f;  // 4 (2^-9 + E 2^-23)
        float e_a = tl.en2[L], e_b = tl.en2[L + 128], q_a = tl.qa2[L];
        for (int j = 0; j < P - 1; ++j) {
            const uint32_t nrm = ring + (uint32_t)(j * part) + (uint32_t)(gown * 32 * p.Rp * 4);
            e_a += lds_f32(nrm + 4u * L);
            e_b += lds_f32(nrm + 4u * (L + 128));
            q_a += lds_f32(nrm + 4u * (kMaxF + L));
        }
        tl.fnorm[L] = sqrtf(e_a) * 1.0001f;
        tl.fnorm[L + 128] = sqrtf(e_b) * 1.0001f;
        tl.qscale[L] = rel * sqrtf(q_a);
    }
    __syncthreads();
    if (rows_here && acc_ok) {
        const float qs = L < p.R ? tl.qscale[L] : 0.f;
        const uint32_t fn = saddr(tl.fnorm);
        const uint32_t stg = ring + (uint32_t)split_out_offset(P, part) + (uint32_t)(warp * kOutBoxBytes * 2);
        bool staged = false;
        for (int g = rank, i = 0; g < G; g += P, ++i) {
            if ((i & 1) != half) continue;
            const int c = 32 * g;
            __syncwarp();
            uint32_t v[32];
            tmem_ld32(tm_rows + (uint32_t)c, v);
            float val[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) val[j] = __uint_as_float(v[j]);
            if (L < p.R) {
                for (int q = 0; q < P - 1; ++q) {
                    const uint32_t pr = ring + (uint32_t)(q * part) + (uint32_t)(((g / P) * 32 * p.Rp + L) * 4);
#pragma unroll
                    for (int j = 0; j < 32; ++j) val[j] += lds_f32(pr + (uint32_t)(j * p.Rp * 4));
                }
            }
            float eps[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) eps[j] = lds_f32(fn + 4u * (c + j));
            // the previous boxes' tensor stores must have read the staging
            if (staged) {
                if (lane == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                __syncwarp();
            }
            // lane = row: its 16-byte chunk q of 8 goes to q ^ (row % 8)
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float lo4[4], hi4[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float e = __fmaf_ru(qs, eps[4 * q + u], 7.9e-31f);
                    lo4[u] = __fsub_rd(val[4 * q + u], e);
                    hi4[u] = __fadd_ru(val[4 * q + u], e);
                }
                const uint32_t at = stg + (uint32_t)(lane * 128 + ((q ^ (lane & 7)) * 16));
                sts_v4(at, lo4[0], lo4[1], lo4[2], lo4[3]);
                sts_v4(at + kOutBoxBytes, hi4[0], hi4[1], hi4[2], hi4[3]);
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            // facts past N and rows past R fall outside the maps: not written
            if (lane == 0) {
                tma_store_2d(&tm_lo, stg, (int)(f0 + c), row0);
                tma_store_2d(&tm_hi, stg + kOutBoxBytes, (int)(f0 + c), row0);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
            staged = true;
        }
        if (lane == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        __syncwarp();
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"((uint32_t)p.tmem_cols)
                     : "memory");
    }
}

// ------------------------------------------------------------------- host

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_encode_mu;

cudaError_t encoder(PFN_cuTensorMapEncodeTiled_v12000 *out)
{
    std::lock_guard<std::mutex> lock(g_encode_mu);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                               cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *out = g_encode;
    return cudaSuccess;
}

// 2-D float32 tensor map over rows of `inner` elements (row pitch `pitch`
// bytes), `outer` rows; boxes of kChunk x box_rows with the 128-byte swizzle.
cudaError_t tmap_f32(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer, uint64_t pitch,
                     uint32_t box_rows)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc;
    cudaError_t e = encoder(&enc);
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {(cuuint32_t)kChunk, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(ptr), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// ---------------------------------------------------- split form: the plan

int split_stages(int F)
{
    const int stage = kSlotQ + F * kChunk * 4;
    return std::max(2, std::min(kMaxStages, kRingBudget / stage));
}

size_t split_smem_bytes(int F)
{
    return 1024 + (size_t)split_stages(F) * (kSlotQ + (size_t)F * kChunk * 4) + sizeof(SplitSmemTail);
}

struct SplitPlan {
    int F = 32, P = 1;
    int64_t tiles = 0;
};

// Facts per tile and CTAs per cluster: the fewest MMAs on any CTA's chain
// (waves of CTAs x chunks per CTA), then the widest tile (fewer CTAs
// reloading the queries).  A cluster's partners must fit CTA 0's ring.
SplitPlan split_plan(int64_t N, int Rp, int E, int sms, int pmax)
{
    const int nk = (E + kChunk - 1) / kChunk;
    SplitPlan best;
    int64_t best_cost = INT64_MAX;
    const int fmax = (int)std::min<int64_t>(kMaxF, (N + 31) / 32 * 32);
    for (int F = fmax; F >= 32; F -= 32) {
        const size_t ring = (size_t)split_stages(F) * (kSlotQ + (size_t)F * kChunk * 4);
        const int64_t tiles = (N + F - 1) / F;
        const int64_t by_sms = std::max<int64_t>(1, sms / tiles);
        int P = (int)std::max<int64_t>(1, std::min<int64_t>({(int64_t)pmax, (int64_t)nk, by_sms}));
        while (P > 1 && split_out_offset(P, split_part_bytes(Rp, F, P)) + kOutStageBytes > ring) --P;
        const int64_t waves = (tiles * P + sms - 1) / sms;
        const int64_t cost = waves * ((nk + P - 1) / P);
        if (cost < best_cost) {
            best_cost = cost;
            best.F = F;
            best.P = P;
            best.tiles = tiles;
        }
    }
    return best;
}

// How many clusters of P CTAs (F facts each) the GPU holds at once: the
// CTAs of a cluster share a GPC, so this can be below SMs / P.  Cached per
// device and shape.
int split_max_clusters(int P, int F)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, P, F);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P);
    cfg.blockDim = dim3(kSplitThreads);
    cfg.dynamicSmemBytes = split_smem_bytes(F);
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)P;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, coarse_split_kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();  // not sticky: the plan falls back to smaller clusters
        n = 0;
    }
    cache[key] = n;
    return n;
}

cudaError_t launch_coarse_split(CoarseParams p, const float *emb, int64_t n_facts, const float *queries,
                                int sms, cudaStream_t s)
{
    cudaError_t e = smem_opt_in(coarse_split_kernel, (int)(1024 + kRingBudget + sizeof(SplitSmemTail)));
    if (e != cudaSuccess) return e;
    SplitPlan pl = split_plan(n_facts, p.Rp, p.E, sms, kMaxSplit);
    while (pl.P > 1 && split_max_clusters(pl.P, pl.F) < pl.tiles)
        pl = split_plan(n_facts, p.Rp, p.E, sms, pl.P - 1);
    p.F = pl.F;
    p.split = pl.P;
    p.mt = 1;
    p.stages = split_stages(pl.F);
    int cols = 32;
    while (cols < pl.F) cols <<= 1;
    p.tmem_cols = cols;
    {
        const int m = p.Rp / 16;
        int d = 1;
        for (int c = 1; c * 16 <= kBoxRowsBMax; ++c)
            if (m % c == 0) d = c;
        p.box_q = 16 * d;
    }
    CUtensorMap te, tq;
    e = tmap_f32(&te, emb, (uint64_t)p.E, (uint64_t)n_facts, (uint64_t)p.E * 4, (uint32_t)split_fact_box(pl.F));
    if (e != cudaSuccess) return e;
    e = tmap_f32(&tq, queries, (uint64_t)p.E, (uint64_t)p.R, (uint64_t)p.E * 4, (uint32_t)p.box_q);
    if (e != cudaSuccess) return e;
    // the interval planes [R][stride] (N facts wide), written as 32 x 32 boxes
    CUtensorMap tlo, thi;
    e = tmap_f32(&tlo, p.lo, (uint64_t)n_facts, (uint64_t)p.R, (uint64_t)p.stride * 4, 32);
    if (e != cudaSuccess) return e;
    e = tmap_f32(&thi, p.hi, (uint64_t)n_facts, (uint64_t)p.R, (uint64_t)p.stride * 4, 32);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(pl.tiles * pl.P));
    cfg.blockDim = dim3(kSplitThreads);
    cfg.dynamicSmemBytes = split_smem_bytes(pl.F);
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)pl.P;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = pl.P > 1 ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, coarse_split_kernel, te, tq, tlo, thi, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

int coarse_stages(int Rp, int mt)
{
    const int per = mt * kStageBytesA + Rp * kChunk * 4;
    return std::max(2, std::min(kMaxStages, kRingBudget / per));
}

size_t coarse_smem_bytes(int Rp, int mt)
{
    const int S = coarse_stages(Rp, mt);
    return 1024 + (size_t)S * (mt * kStageBytesA + (size_t)Rp * kChunk * 4) + sizeof(CoarseSmemTail);
}

cudaError_t launch_coarse(const CoarseParams &p0, const float *emb, int64_t n_facts, const float *queries,
                          cudaStream_t s)
{
    CoarseParams p = p0;
    DeviceInfo di;
    cudaError_t e0 = device_info(&di);
    if (e0 != cudaSuccess) return e0;
    // up to 128 queries: queries on M, facts on N, K split over a cluster
    if (p.Rp <= kQTile) return launch_coarse_split(p, emb, n_facts, queries, di.sms, s);
    // more: facts on M, all queries on N (<= 256); two accumulators per CTA
    // (256 facts sharing each query chunk) once the tiles of 256 still fill
    // the GPU, one otherwise
    const int64_t tiles128 = (n_facts + kTileM - 1) / kTileM;
    p.mt = tiles128 >= 2 * (int64_t)di.sms ? 2 : 1;
    p.stages = coarse_stages(p.Rp, p.mt);
    int cols = 32;
    while (cols < p.Rp) cols <<= 1;
    p.tmem_cols = cols * p.mt;  // <= 512: cols <= 256
    CUtensorMap te, tq;
    cudaError_t e = tmap_f32(&te, emb, (uint64_t)p.E, (uint64_t)n_facts, (uint64_t)p.E * 4, kBoxRowsA);
    if (e != cudaSuccess) return e;
    // query rows per box: 16 x the largest divisor d <= 8 of Rp / 16, so that
    // the boxes tile the Rp padded rows of a stage exactly
    {
        const int m = p.Rp / 16;
        int d = 1;
        for (int c = 1; c * 16 <= kBoxRowsBMax; ++c)
            if (m % c == 0) d = c;
        p.box_q = 16 * d;
    }
    e = tmap_f32(&tq, queries, (uint64_t)p.E, (uint64_t)p.R, (uint64_t)p.E * 4, (uint32_t)p.box_q);
    if (e != cudaSuccess) return e;
    const size_t smem = coarse_smem_bytes(p.Rp, p.mt);
    // the opt-in is made once per device, so it covers the largest ring any
    // query count needs
    size_t most = 0;
    for (int rp = 16; rp <= KVI_MAX_SHARED_QUERIES; rp += 16)
        most = std::max(most, std::max(coarse_smem_bytes(rp, 1), coarse_smem_bytes(rp, 2)));
    e = smem_opt_in(coarse_kernel, (int)most);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)((n_facts + (int64_t)p.mt * kTileM - 1) / ((int64_t)p.mt * kTileM));
    coarse_kernel<<<grid, kCoarseThreads, smem, s>>>(te, tq, p);
    return cudaGetLastError();
}

}  // namespace kvi

#ifdef KVI_DEBUG_CHECKS
#include "kvi_debug.h"

extern "C" kvi_status kvi_debug_stall_coarse_chunk(int32_t cta, int32_t chunk)
{
    const int c = cta < 0 ? -1 : (int)cta, k = cta < 0 ? -1 : (int)chunk;
    cudaError_t e = cudaMemcpyToSymbol(kvi::g_debug_stall_cta, &c, sizeof c);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(kvi::g_debug_stall_chunk, &k, sizeof k);
    if (e != cudaSuccess) return kvi::set_error(KVI_ERR_CUDA, cudaGetErrorString(e));
    return KVI_OK;
}
#endif

// kvi_shared.cu -- many queries against one shared fact store.
//
// "InferScale: GPU-Native KV Injection for Personalized LLM Serving",
// Section 6.4: concurrent users issue queries against one conversation's
// memory store.  Scoring R queries against the same N x E embedding matrix
// is a dense contraction S = Q E^T, so here it runs on the 5th-generation
// tensor cores instead of R separate scans of the matrix:
//
//   coarse_kernel   one CTA per 128 facts.  A TMA producer warp (one box per
//                   lane) streams the facts' rows and all queries through a
//                   ring of 128-byte swizzled stages; one thread issues
//                   tcgen05.mma (kind::tf32,
//                   M = 128, N = R padded to 16) accumulating in tensor
//                   memory; four warps compute the row norms from the same
//                   stages and, at the end, read the accumulator back
//                   (tcgen05.ld) and write an interval [lo, hi] that provably
//                   holds every exact score (bound below).
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

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "kvi_internal.cuh"

namespace kvi {
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
        for (int kc = 0; kc < nk; ++kc) {
            const int s = kc % S;
            const int round = kc / S;
            bool go = true;
            if (lane == 0 && round > 0) go = wait_bar(saddr(&tl.empty[s]), (uint32_t)((round - 1) & 1));
            if (!__shfl_sync(0xffffffffu, go ? 1 : 0, 0)) {
                if (lane == 0) record_status(p.status, KVI_ERR_TIMEOUT);
                ok = false;
                break;
            }
            const uint32_t fb = saddr(&tl.full[s]);
            if (lane == 0) {
                if (round > 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb), "r"(bytes) : "memory");
            }
            __syncwarp();
            for (int j = lane; j < na + nb; j += 32) {
                if (j < na)
                    tma_2d(saddr(a_st + (size_t)s * stage_a + (size_t)j * kBoxRowsA * 128), &tm_emb,
                           kc * kChunk, tile * MT * kTileM + j * kBoxRowsA, fb);
                else
                    tma_2d(saddr(b_st + (size_t)s * stage_b + (size_t)(j - na) * bq * 128), &tm_q,
                           kc * kChunk, (j - na) * bq, fb);
            }
            issued = kc + 1;
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
            for (int kc = 0; kc < nk; ++kc) {
                const int s = kc % S;
                if (!wait_bar(saddr(&tl.full[s]), (uint32_t)((kc / S) & 1))) {
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
        for (int kc = 0; kc < nk; ++kc) {
            const int s = kc % S;
            const bool got = wait_bar(saddr(&tl.full[s]), (uint32_t)((kc / S) & 1));
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
    // two accumulators per CTA (256 facts sharing each query chunk) once the
    // tiles of 256 still fill the GPU; one otherwise
    DeviceInfo di;
    cudaError_t e0 = device_info(&di);
    if (e0 != cudaSuccess) return e0;
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

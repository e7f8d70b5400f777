// kvi_retrieve.cu -- retrieval side of the retrieve-and-inject path.
//
// "InferScale: GPU-Native KV Injection for Personalized LLM Serving", Figure 2
// caption: the fact store keeps a retrieval embedding per fact_id and, at
// serving time, the top-k facts for the query are resolved to their KV and
// positioned.  The paper searches an approximate GPU index; this library
// computes the exact top-k by a full scan, which is HBM-bound (every
// embedding row is read once per query), so the kernels here are shaped for
// bandwidth, not for tensor cores:
//
//   score_kernel   one warp per fact row, 16-byte streaming loads, query held
//                  in registers; the dot product is accumulated with Dot2
//                  (Ogita, Rump & Oishi, "Accurate Sum and Dot Product", SIAM
//                  J. Sci. Comput. 26(6), 2005: error-free TwoProduct by FMA
//                  and TwoSum, carried as a float32 pair) and the pair is
//                  turned into a float64 selection key.  Each key also bumps a
//                  4096-bucket histogram of its float32 rounding, a monotone
//                  map, so the selector knows which bucket holds the k-th key.
//   select_kernel  one CTA per request: buckets above the k-th one are taken
//                  whole; the k-th bucket's keys are ranked exactly (or, when
//                  it is crowded, refined by an 8-bit radix select on the full
//                  64-bit key, down to ties, which go to the lower fact id).
//                  In the fused path it also places the facts (rank order,
//                  back to back from the request's start) and publishes the
//                  request's token count; the last CTA to finish turns those
//                  counts into request offsets for the inject kernel.
//   place_kernel   placement alone, for the split API.
#include <cuda_runtime.h>

#include "kvi_internal.cuh"

namespace kvi {
namespace {

__device__ __forceinline__ void record(int32_t *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// 16-byte load that bypasses L1 allocation: each embedding row is read once.
__device__ __forceinline__ float4 ld_stream_f4(const float4 *p)
{
    float4 v;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// TwoSum (Knuth): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// One Dot2 step: add x*y to the pair (s, c) with TwoProduct + TwoSum.
__device__ __forceinline__ void dot2_step(float x, float y, float &s, float &c)
{
    const float pr = __fmul_rn(x, y);
    const float pe = __fmaf_rn(x, y, -pr);
    float ns, se;
    two_sum(s, pr, ns, se);
    s = ns;
    c = __fadd_rn(c, __fadd_rn(se, pe));
}

__device__ __forceinline__ void dot2_f4(const float4 &q, const float4 &e, float &s, float &c)
{
    dot2_step(q.x, e.x, s, c);
    dot2_step(q.y, e.y, s, c);
    dot2_step(q.z, e.z, s, c);
    dot2_step(q.w, e.w, s, c);
}

// Butterfly reduction of (s, c) pairs across the warp, compensated.
__device__ __forceinline__ void warp_reduce_pair(float &s, float &c)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
        const float c2 = __shfl_xor_sync(0xffffffffu, c, off);
        float ns, e;
        two_sum(s, s2, ns, e);
        s = ns;
        c = __fadd_rn(__fadd_rn(c, c2), e);
    }
}

// Order-preserving map double -> uint64 (larger key = larger score).  -0 is
// folded onto +0 first so that the two compare equal, as they do as doubles.
__device__ __forceinline__ uint64_t order_key(double s)
{
    s = __dadd_rn(s, 0.0);
    const uint64_t u = (uint64_t)__double_as_longlong(s);
    return (u >> 63) ? ~u : (u | 0x8000000000000000ull);
}

__device__ __forceinline__ double unorder_key(uint64_t u)
{
    const uint64_t v = (u >> 63) ? (u & 0x7fffffffffffffffull) : ~u;
    return __longlong_as_double((long long)v);
}

// First-level bucket: top 12 bits of the order-preserving image of the key
// rounded to float32.  Rounding is monotone, so key_a > key_b implies
// bucket_a >= bucket_b.
__device__ __forceinline__ uint32_t bucket_of(uint64_t okey)
{
    const float f = __fadd_rn(__double2float_rn(unorder_key(okey)), 0.0f);
    uint32_t u = __float_as_uint(f);
    u = (u >> 31) ? ~u : (u | 0x80000000u);
    return u >> 20;
}

__device__ __forceinline__ bool better(uint64_t ka, int32_t ia, uint64_t kb, int32_t ib)
{
    return ka > kb || (ka == kb && ia < ib);
}

__device__ __forceinline__ bool store_ok(const kvi_store_view &st, const kvi_geometry &g,
                                         int64_t max_facts, int32_t k)
{
    return st.g.layers == g.layers && st.g.kv_heads == g.kv_heads &&
           st.g.head_dim == g.head_dim && st.g.embed_dim == g.embed_dim &&
           st.n_facts >= k && st.n_facts <= max_facts && st.n_facts <= 0x7fffffff &&
           st.n_tokens >= 0 && st.kv != nullptr && st.emb != nullptr &&
           st.fact_start != nullptr && st.fact_len != nullptr &&
           (((uintptr_t)st.emb) & 15) == 0 && (((uintptr_t)st.kv) & 15) == 0;
}

__device__ __forceinline__ kvi_store_view load_store(const StoreRef &s, int r)
{
    return s.many ? s.many[r] : s.single;
}

// ------------------------------------------------------------------ scoring

template <int NV>  // float4 per lane per row (E = 128 * NV); 0 = any E % 4 == 0
__global__ void __launch_bounds__(kScoreThreads)
score_kernel(const __grid_constant__ ScoreParams p)
{
    const int r = blockIdx.y;
    const kvi_store_view st = load_store(p.store, r);
    if (p.store.many && !store_ok(st, p.g, p.max_facts, 1)) return;  // reported by select
    const int64_t N = st.n_facts;
    const int64_t row0 = (int64_t)blockIdx.x * p.rows_per_cta;
    if (row0 >= N) return;
    const int64_t row1 = min(N, row0 + (int64_t)p.rows_per_cta);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int E = p.g.embed_dim;
    const float4 *q4 = reinterpret_cast<const float4 *>(p.queries + (int64_t)r * E);
    uint64_t *keys = p.keys + (int64_t)r * p.key_stride;
    uint32_t *hist = p.hist + (int64_t)r * kHistBins;

    float4 qv[NV > 0 ? NV : 1];
    if constexpr (NV > 0) {
#pragma unroll
        for (int m = 0; m < NV; ++m) qv[m] = __ldg(q4 + lane + 32 * m);
    }
    for (int64_t i = row0 + warp; i < row1; i += kScoreThreads / 32) {
        const float4 *e4 = reinterpret_cast<const float4 *>(st.emb + i * E);
        float s = 0.f, c = 0.f;
        if constexpr (NV > 0) {
            float4 ev[NV];
#pragma unroll
            for (int m = 0; m < NV; ++m) ev[m] = ld_stream_f4(e4 + lane + 32 * m);
#pragma unroll
            for (int m = 0; m < NV; ++m) dot2_f4(qv[m], ev[m], s, c);
        } else {
            for (int v = lane; v < E / 4; v += 32) dot2_f4(__ldg(q4 + v), ld_stream_f4(e4 + v), s, c);
        }
        warp_reduce_pair(s, c);
        if (lane == 0) {
            const uint64_t ok = order_key(__dadd_rn((double)s, (double)c));
            keys[i] = ok;
            atomicAdd(hist + bucket_of(ok), 1u);
        }
    }
}

// ---------------------------------------------------------------- selection

// Inclusive scan of one value per thread over a 1024-thread block.
__device__ __forceinline__ uint32_t block_incl_scan(uint32_t v, uint32_t *warp_tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    const uint32_t before = warp ? warp_tot[warp - 1] : 0u;
    __syncthreads();  // warp_tot is reused by the next call
    return v + before;
}

// Same for 64-bit values (request token offsets).
__device__ __forceinline__ uint64_t block_incl_scan64(uint64_t v, uint64_t *warp_tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        uint64_t w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    const uint64_t before = warp ? warp_tot[warp - 1] : 0ull;
    __syncthreads();
    return v + before;
}

struct SelectSmem {
    uint32_t hist[kHistBins];
    uint64_t cand_key[kCandCap];
    int32_t cand_id[kCandCap];
    uint64_t sure_key[KVI_MAX_K];
    int32_t sure_id[KVI_MAX_K];
    uint64_t out_key[KVI_MAX_K];
    int32_t out_id[KVI_MAX_K];
    int32_t out_len[KVI_MAX_K];
    uint32_t warp_tot[32];
    uint64_t warp_tot64[32];
    uint32_t n_sure, n_cand, bucket, above, digit, above2;
    int32_t last;
    int32_t fit;
};

// Rank the n_cand candidates in shared memory and move the best `need` of
// them to the sure list (positions base .. base + need).
__device__ void take_best_candidates(SelectSmem &sm, uint32_t n_cand, uint32_t need, uint32_t base)
{
    for (uint32_t c = threadIdx.x; c < n_cand; c += kSelectThreads) {
        const uint64_t kc = sm.cand_key[c];
        const int32_t ic = sm.cand_id[c];
        uint32_t rank = 0;
        for (uint32_t o = 0; o < n_cand; ++o) rank += better(sm.cand_key[o], sm.cand_id[o], kc, ic);
        if (rank < need && base + rank < (uint32_t)KVI_MAX_K) {
            sm.sure_key[base + rank] = kc;
            sm.sure_id[base + rank] = ic;
        }
    }
}

__global__ void __launch_bounds__(kSelectThreads, 1)
select_kernel(const __grid_constant__ SelectParams p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SelectSmem &sm = *reinterpret_cast<SelectSmem *>(smem_raw);
    const int r = blockIdx.x;
    const int tid = threadIdx.x;
    const int32_t k = p.k;
    const kvi_store_view st = load_store(p.store, r);
    const bool ok = !p.store.many || store_ok(st, p.g, p.max_facts, k);
    const int64_t N = st.n_facts;
    const uint64_t *keys = p.keys + (int64_t)r * p.key_stride;

    if (ok) {
        // 1. the bucket holding the k-th key, from the histogram (bucket
        //    4095 is the best); thread t owns buckets 4095-4t .. 4092-4t.
        const uint32_t *gh = p.hist + (int64_t)r * kHistBins;
        const int top = kHistBins - 1 - 4 * tid;
        const uint32_t c0 = __ldcg(gh + top), c1 = __ldcg(gh + top - 1);
        const uint32_t c2 = __ldcg(gh + top - 2), c3 = __ldcg(gh + top - 3);
        const uint32_t incl = block_incl_scan(c0 + c1 + c2 + c3, sm.warp_tot);
        const uint32_t excl = incl - (c0 + c1 + c2 + c3);
        if (tid == 0) { sm.n_sure = 0; sm.n_cand = 0; }
        for (int e = tid; e < KVI_MAX_K; e += kSelectThreads) {
            sm.sure_key[e] = 0;
            sm.sure_id[e] = -1;
        }
        if (excl < (uint32_t)k && incl >= (uint32_t)k) {
            const uint32_t cs[4] = {c0, c1, c2, c3};
            uint32_t run = excl;
            for (int j = 0; j < 4; ++j) {
                if (run + cs[j] >= (uint32_t)k) {
                    sm.bucket = (uint32_t)(top - j);
                    sm.above = run;
                    sm.hist[0] = cs[j];  // population of the k-th bucket
                    break;
                }
                run += cs[j];
            }
        }
        __syncthreads();
        const uint32_t b0 = sm.bucket;
        const uint32_t above = sm.above;
        const uint32_t M = sm.hist[0];
        const uint32_t need = (uint32_t)k - above;

        // 2. keys above the bucket are in; keys in it are candidates.
        for (int64_t i = tid; i < N; i += kSelectThreads) {
            const uint64_t key = __ldcg(keys + i);
            const uint32_t b = bucket_of(key);
            if (b > b0) {
                const uint32_t at = atomicAdd(&sm.n_sure, 1u);
                if (at < (uint32_t)KVI_MAX_K) { sm.sure_key[at] = key; sm.sure_id[at] = (int32_t)i; }
            } else if (b == b0 && M <= (uint32_t)kCandCap) {
                const uint32_t at = atomicAdd(&sm.n_cand, 1u);
                if (at < (uint32_t)kCandCap) { sm.cand_key[at] = key; sm.cand_id[at] = (int32_t)i; }
            }
        }
        __syncthreads();

        if (M <= (uint32_t)kCandCap) {
            take_best_candidates(sm, M, need, above);
        } else {
            // 3. crowded bucket: radix select on the 64-bit key, 8 bits at a
            //    time, restricted to bucket b0.
            uint64_t prefix = 0;
            uint32_t need_r = need;
            bool done = false;
            for (int shift = 56; shift >= 0 && !done; shift -= 8) {
                for (int b = tid; b < 256; b += kSelectThreads) sm.hist[b] = 0;
                __syncthreads();
                for (int64_t i = tid; i < N; i += kSelectThreads) {
                    const uint64_t key = __ldcg(keys + i);
                    if (bucket_of(key) != b0) continue;
                    if (shift < 56 && (key >> (shift + 8)) != prefix) continue;
                    atomicAdd(&sm.hist[(key >> shift) & 0xff], 1u);
                }
                __syncthreads();
                if (tid == 0) {
                    uint32_t run = 0;
                    for (int d = 255; d >= 0; --d) {
                        if (run + sm.hist[d] >= need_r) { sm.digit = (uint32_t)d; sm.above2 = run; break; }
                        run += sm.hist[d];
                    }
                }
                __syncthreads();
                const uint32_t dd = sm.digit;
                const uint32_t above2 = sm.above2;
                const uint32_t M2 = sm.hist[dd];
                // keys of the current prefix with a larger digit are in
                for (int64_t i = tid; i < N; i += kSelectThreads) {
                    const uint64_t key = __ldcg(keys + i);
                    if (bucket_of(key) != b0) continue;
                    if (shift < 56 && (key >> (shift + 8)) != prefix) continue;
                    if (((key >> shift) & 0xff) > dd) {
                        const uint32_t at = atomicAdd(&sm.n_sure, 1u);
                        if (at < (uint32_t)KVI_MAX_K) { sm.sure_key[at] = key; sm.sure_id[at] = (int32_t)i; }
                    }
                }
                need_r -= above2;
                prefix = (prefix << 8) | dd;
                if (tid == 0) sm.n_cand = 0;
                __syncthreads();
                if (M2 <= (uint32_t)kCandCap) {
                    for (int64_t i = tid; i < N; i += kSelectThreads) {
                        const uint64_t key = __ldcg(keys + i);
                        if (bucket_of(key) != b0 || (key >> shift) != prefix) continue;
                        const uint32_t at = atomicAdd(&sm.n_cand, 1u);
                        if (at < (uint32_t)kCandCap) { sm.cand_key[at] = key; sm.cand_id[at] = (int32_t)i; }
                    }
                    __syncthreads();
                    const uint32_t base = sm.n_sure;
                    take_best_candidates(sm, M2, need_r, base);
                    done = true;
                }
                __syncthreads();
            }
            if (!done) {
                // every remaining key equals `prefix`: the lowest ids win.
                const uint32_t base = sm.n_sure;
                uint32_t taken = 0;
                for (int64_t i0 = 0; i0 < N && taken < need_r; i0 += kSelectThreads) {
                    const int64_t i = i0 + tid;
                    uint32_t flag = 0;
                    uint64_t key = 0;
                    if (i < N) {
                        key = __ldcg(keys + i);
                        flag = (bucket_of(key) == b0 && key == prefix) ? 1u : 0u;
                    }
                    const uint32_t incl2 = block_incl_scan(flag, sm.warp_tot);
                    const uint32_t at = taken + incl2 - flag;
                    if (flag && at < need_r && base + at < (uint32_t)KVI_MAX_K) {
                        sm.sure_key[base + at] = key;
                        sm.sure_id[base + at] = (int32_t)i;
                    }
                    taken += sm.warp_tot[31];  // block total of flags
                    __syncthreads();
                }
            }
        }
        __syncthreads();

        // 4. sort the k selected keys into rank order.
        for (int e = tid; e < k; e += kSelectThreads) {
            const uint64_t ke = sm.sure_key[e];
            const int32_t ie = sm.sure_id[e];
            int rank = 0;
            for (int o = 0; o < k; ++o) rank += better(sm.sure_key[o], sm.sure_id[o], ke, ie);
            sm.out_key[rank] = ke;
            sm.out_id[rank] = ie;
        }
        __syncthreads();
    }

    for (int j = tid; j < k; j += kSelectThreads) {
        p.ids[(int64_t)r * k + j] = ok ? sm.out_id[j] : -1;
        p.scores[(int64_t)r * k + j] = ok ? __double2float_rn(unorder_key(sm.out_key[j])) : __int_as_float(0x7fc00000);
    }
    if (!p.place) return;

    // 5. placement: rank order, back to back from the request's start.
    if (!ok && tid == 0) record(p.status, KVI_ERR_OUT_OF_RANGE);
    for (int j = tid; j < k; j += kSelectThreads) {
        int32_t len = 0;
        if (ok) {
            const int32_t f = sm.out_id[j];
            if (f >= 0 && (int64_t)f < N) {
                const int64_t s0 = st.fact_start[f];
                const int32_t l0 = st.fact_len[f];
                if (l0 >= 0 && s0 >= 0 && s0 + l0 <= st.n_tokens) len = l0;
                else record(p.status, KVI_ERR_OUT_OF_RANGE);
            } else {
                record(p.status, KVI_ERR_OUT_OF_RANGE);
            }
        }
        sm.out_len[j] = len;
    }
    __syncthreads();
    if (tid == 0) {
        const int64_t start = p.start_pos[r];
        const int32_t tl = p.table_lens[r];
        int64_t run = 0;
        for (int j = 0; j < k; ++j) {
            p.cum[(int64_t)r * (k + 1) + j] = (int32_t)run;
            p.pos[(int64_t)r * k + j] = (int32_t)(start + run);
            run += sm.out_len[j];
        }
        p.cum[(int64_t)r * (k + 1) + k] = (int32_t)run;
        int fit = 1;
        if (tl < 0 || tl > p.max_blocks) { record(p.status, KVI_ERR_OUT_OF_RANGE); fit = 0; }
        else if (start < 0 || start + run > (int64_t)tl * p.block_size) { record(p.status, KVI_ERR_CAPACITY); fit = 0; }
        p.tok[r] = fit && ok ? run : 0;
        __threadfence();
        const uint32_t prev = atomicAdd(p.counter, 1u);
        sm.last = (prev == (uint32_t)(p.R - 1));
    }
    __syncthreads();
    if (!sm.last) return;
    // 6. last CTA: request token offsets (exclusive prefix over requests).
    __threadfence();
    int64_t carry = 0;
    for (int r0 = 0; r0 < p.R; r0 += kSelectThreads) {
        const int rr = r0 + tid;
        const uint64_t t = rr < p.R ? (uint64_t)__ldcg(p.tok + rr) : 0ull;
        const uint64_t incl2 = block_incl_scan64(t, sm.warp_tot64);
        if (rr < p.R) p.req_off[rr] = carry + (int64_t)(incl2 - t);
        carry += (int64_t)sm.warp_tot64[31];
        __syncthreads();
    }
    if (tid == 0) p.req_off[p.R] = carry;
}

// ---------------------------------------------------------------- placement

__global__ void __launch_bounds__(256) place_kernel(const __grid_constant__ PlaceParams p)
{
    __shared__ int32_t lens[KVI_MAX_K];
    for (int j = threadIdx.x; j < p.n; j += blockDim.x) {
        const int32_t f = p.ids[j];
        int32_t len = 0;
        if (f >= 0 && (int64_t)f < p.store.n_facts) len = max(0, p.store.fact_len[f]);
        else record(p.status, KVI_ERR_OUT_OF_RANGE);
        lens[j] = len;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t run = p.start;
        for (int j = 0; j < p.n; ++j) {
            p.pos[j] = (int32_t)run;
            run += lens[j];
        }
        if (run > 0x7fffffff) record(p.status, KVI_ERR_OUT_OF_RANGE);
    }
}

template <int NV>
cudaError_t launch_score_nv(const ScoreParams &p, cudaStream_t s)
{
    const unsigned gx = (unsigned)((p.max_facts + p.rows_per_cta - 1) / p.rows_per_cta);
    score_kernel<NV><<<dim3(gx, (unsigned)p.R), kScoreThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score(const ScoreParams &p, cudaStream_t s)
{
    const int E = p.g.embed_dim;
    if (E % 128 == 0) {
        switch (E / 128) {
        case 1: return launch_score_nv<1>(p, s);
        case 2: return launch_score_nv<2>(p, s);
        case 3: return launch_score_nv<3>(p, s);
        case 4: return launch_score_nv<4>(p, s);
        case 6: return launch_score_nv<6>(p, s);
        case 8: return launch_score_nv<8>(p, s);
        case 12: return launch_score_nv<12>(p, s);
        case 16: return launch_score_nv<16>(p, s);
        default: break;
        }
    }
    return launch_score_nv<0>(p, s);
}

cudaError_t launch_select(const SelectParams &p, cudaStream_t s)
{
    static_assert(sizeof(SelectSmem) <= 227 * 1024, "select smem");
    const int smem = (int)sizeof(SelectSmem);
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    select_kernel<<<(unsigned)p.R, kSelectThreads, smem, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_place(const PlaceParams &p, cudaStream_t s)
{
    place_kernel<<<1, 256, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvi

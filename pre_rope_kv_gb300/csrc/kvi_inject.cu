// kvi_inject.cu -- gather, Chunked-RoPE rotate and paged scatter.
//
// "InferScale: GPU-Native KV Injection for Personalized LLM Serving":
// Section 5.1 / Theorem 6 (Chunked RoPE) -- each fact's keys are stored before
// rotary encoding and rotated to the positions they take in the prompt when
// injected; Section 3.4 -- K and V are scatter-copied into the engine's paged
// blocks before the forward pass, so only the query is prefilled.
//
// The kernel is a pure HBM stream: every injected byte is read once from the
// store and written once to the pool.  It is persistent (one wave of CTAs,
// grid-stride over work items) because the number of tokens is only known on
// the device in the fused path.  A work item is one 2 x 16-byte vector pair
// of one head row, for one token, K or V, over a group of kLayerGroup layers:
//
//   - the two vectors of a pair are elements [8v, 8v+8) and [D/2+8v, D/2+8v+8)
//     of a head, i.e. the rotate-half partners, so the rotation needs no
//     data exchange between threads;
//   - consecutive threads take consecutive pairs of the same row, so each
//     warp reads and writes whole 128-byte lines of the store and the page;
//   - the cos/sin entries of the token's position are loaded once per item
//     and reused across its layers.
//
// Rotation accuracy.  The table holds cos and sin of p * omega_i computed in
// float64 on the host, split into a 16-significant-bit head and a float32
// tail.  A bf16 key has 8 significant bits, so x * head is exact in float32,
// and y = fma(x_i, c_hi, -x_j * s_hi) + (x_i * c_lo - x_j * s_lo) is within a
// few float32 ulps of the exact rotation at any position; one rounding to
// bf16 follows.  Position 0 is the identity and copies the key bits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kvi_internal.cuh"

namespace kvi {
namespace {

__device__ __forceinline__ void record(int32_t *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint4 ld_stream_u4(const void *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_u4(void *p, const uint4 &v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half)
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Rotate 8 rotate-half pairs: lo holds x_i, hi holds x_{i+D/2}.
__device__ __forceinline__ void rotate8(uint4 &lo, uint4 &hi, const float4 *cs)
{
    uint32_t *pl = reinterpret_cast<uint32_t *>(&lo);
    uint32_t *ph = reinterpret_cast<uint32_t *>(&hi);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        float y0[2], y1[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float x0 = h ? bf_hi(pl[w]) : bf_lo(pl[w]);
            const float x1 = h ? bf_hi(ph[w]) : bf_lo(ph[w]);
            const float4 t = cs[2 * w + h];  // {cos_hi, cos_lo, sin_hi, sin_lo}
            y0[h] = __fadd_rn(__fmaf_rn(x0, t.x, -__fmul_rn(x1, t.z)),
                              __fsub_rn(__fmul_rn(x0, t.y), __fmul_rn(x1, t.w)));
            y1[h] = __fadd_rn(__fmaf_rn(x1, t.x, __fmul_rn(x0, t.z)),
                              __fadd_rn(__fmul_rn(x1, t.y), __fmul_rn(x0, t.w)));
        }
        pl[w] = pack_bf16(y0[0], y0[1]);
        ph[w] = pack_bf16(y1[0], y1[1]);
    }
}

// Largest j in [0, n) with a[j] <= x, for non-decreasing a[0..n] and
// a[0] <= x < a[n].
template <typename T, typename U>
__device__ __forceinline__ int search_le(const T *a, int n, U x)
{
    int lo = 0, hi = n;  // invariant: a[lo] <= x < a[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((U)a[mid] <= x) lo = mid; else hi = mid;
    }
    return lo;
}

template <typename T, typename U>
__device__ __forceinline__ int search_le_cg(const T *a, int n, U x)
{
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((U)__ldcg(a + mid) <= x) lo = mid; else hi = mid;
    }
    return lo;
}

__global__ void __launch_bounds__(kInjectThreads)
inject_kernel(const __grid_constant__ InjectParams p)
{
    __shared__ int32_t s_cum[KVI_MAX_INJECT_FACTS + 1];
    __shared__ int32_t s_part[kInjectThreads];

    int64_t T;
    if (!p.fused) {
        // token prefix of the n facts (invalid ids or extents count as 0)
        const kvi_store_view &st = p.store.single;
        constexpr int per = (KVI_MAX_INJECT_FACTS + kInjectThreads - 1) / kInjectThreads;
        const int j0 = threadIdx.x * per;
        int32_t run = 0;
        for (int j = j0; j < j0 + per && j < p.n; ++j) {
            const int32_t f = p.ids[j];
            int32_t len = 0;
            if (f >= 0 && (int64_t)f < st.n_facts) {
                const int64_t s0 = st.fact_start[f];
                const int32_t l0 = st.fact_len[f];
                if (l0 >= 0 && s0 >= 0 && s0 + l0 <= st.n_tokens) len = l0;
                else if (blockIdx.x == 0) record(p.status, KVI_ERR_OUT_OF_RANGE);
            } else if (blockIdx.x == 0) {
                record(p.status, KVI_ERR_OUT_OF_RANGE);
            }
            s_cum[j + 1] = len;  // length for now, prefix below
            run += len;
        }
        s_part[threadIdx.x] = run;
        __syncthreads();
        if (threadIdx.x == 0) {
            int32_t acc = 0;
            for (int t = 0; t < kInjectThreads; ++t) {
                const int32_t v = s_part[t];
                s_part[t] = acc;
                acc += v;
            }
        }
        __syncthreads();
        int32_t acc = s_part[threadIdx.x];
        if (threadIdx.x == 0) s_cum[0] = 0;
        for (int j = j0; j < j0 + per && j < p.n; ++j) {
            acc += s_cum[j + 1];
            s_cum[j + 1] = acc;
        }
        __syncthreads();
        T = s_cum[p.n];
    } else {
        T = __ldcg(p.req_off + p.R);
    }

    const int D = p.D, H = p.H, L = p.L, B = p.block_size;
    const int half = D >> 1;
    const int vph = D >> 4;  // vector pairs per head
    const int VP = H * vph;  // vector pairs per token row
    const int NG = (L + kLayerGroup - 1) / kLayerGroup;
    const int64_t HD = (int64_t)H * D;
    const int64_t W = T * 2 * NG * VP;

    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < W;
         w += (int64_t)gridDim.x * blockDim.x) {
        int64_t rest = w / VP;
        const int qq = (int)(w - rest * VP);
        const int kvsel = (int)(rest & 1);
        rest >>= 1;
        const int64_t tok = rest / NG;
        const int g = (int)(rest - tok * NG);

        // which fact and which of its tokens
        int32_t f;
        int64_t pos;
        const int32_t *bt;
        int32_t tlen;
        int64_t row;
        const void *kvbase;
        int64_t n_tokens;
        if (!p.fused) {
            const int j = search_le(s_cum, p.n, (int32_t)tok);
            const int32_t t = (int32_t)tok - s_cum[j];
            f = p.ids[j];
            pos = (int64_t)p.pos[j] + t;
            bt = p.block_tables;
            tlen = p.table_len;
            row = p.store.single.fact_start[f] + t;
            kvbase = p.store.single.kv;
            n_tokens = p.store.single.n_tokens;
        } else {
            const int r = search_le_cg(p.req_off, p.R, tok);
            const int32_t local = (int32_t)(tok - __ldcg(p.req_off + r));
            const int32_t *cumr = p.cum + (int64_t)r * (p.k + 1);
            const int j = search_le_cg(cumr, p.k, local);
            const int32_t t = local - __ldcg(cumr + j);
            f = __ldcg(p.ids + (int64_t)r * p.k + j);
            pos = (int64_t)__ldcg(p.pos + (int64_t)r * p.k + j) + t;
            bt = p.block_tables + (int64_t)r * p.max_blocks;
            tlen = p.table_lens[r];
            const kvi_store_view *sv = p.store.many + r;
            row = sv->fact_start[f] + t;
            kvbase = sv->kv;
            n_tokens = sv->n_tokens;
        }

        // where it goes
        if (pos < 0 || pos >= (int64_t)tlen * B || pos >= p.rope_positions) {
            record(p.status, KVI_ERR_OUT_OF_RANGE);
            continue;
        }
        const int32_t blk = bt[pos / B];
        const int32_t off = (int32_t)(pos % B);
        if (blk < 0 || blk >= p.num_blocks) {
            record(p.status, KVI_ERR_OUT_OF_RANGE);
            continue;
        }

        const int h = qq / vph;
        const int v = qq - h * vph;
        const int64_t e_lo = (int64_t)h * D + 8 * v;
        const int64_t e_hi = e_lo + half;
        const bool rot = (kvsel == 0) && (pos != 0);

        float4 cs[8];
        if (rot) {
            const float4 *tp = p.rope + pos * half + 8 * v;
#pragma unroll
            for (int e = 0; e < 8; ++e) cs[e] = __ldg(tp + e);
        }

        const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(kvbase) +
                                   ((int64_t)kvsel * n_tokens + row) * HD;
        const int64_t lstride = 2 * n_tokens * HD;  // elements between layers
        const int64_t dst_off = (((int64_t)kvsel * p.num_blocks + blk) * B + off) * HD;
        const int l0 = g * kLayerGroup;
        const int l1 = min(L, l0 + kLayerGroup);
        int l = l0;
        for (; l + 4 <= l1; l += 4) {
            uint4 a[4], b[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const __nv_bfloat16 *s = src + (int64_t)(l + u) * lstride;
                a[u] = ld_stream_u4(s + e_lo);
                b[u] = ld_stream_u4(s + e_hi);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (rot) rotate8(a[u], b[u], cs);
                __nv_bfloat16 *d = reinterpret_cast<__nv_bfloat16 *>(p.layer_base[l + u]) + dst_off;
                st_u4(d + e_lo, a[u]);
                st_u4(d + e_hi, b[u]);
            }
        }
        for (; l < l1; ++l) {
            const __nv_bfloat16 *s = src + (int64_t)l * lstride;
            uint4 a = ld_stream_u4(s + e_lo);
            uint4 b = ld_stream_u4(s + e_hi);
            if (rot) rotate8(a, b, cs);
            __nv_bfloat16 *d = reinterpret_cast<__nv_bfloat16 *>(p.layer_base[l]) + dst_off;
            st_u4(d + e_lo, a);
            st_u4(d + e_hi, b);
        }
    }
}

}  // namespace

cudaError_t launch_inject(const InjectParams &p, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(di.sms * di.inject_ctas_per_sm);
    inject_kernel<<<grid, kInjectThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t inject_occupancy(int *ctas_per_sm)
{
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, inject_kernel, kInjectThreads, 0);
}

}  // namespace kvi

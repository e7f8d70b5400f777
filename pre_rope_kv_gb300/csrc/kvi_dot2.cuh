// Compensated dot products (Dot2) and the 64-bit order keys of their
// results, shared by every kernel that scores facts, so that the scan, the
// shared-store rescore and the graph search rank facts by identical keys.
//
// Dot2 is the Ogita-Rump-Oishi accurate dot product (TwoProduct by fma plus
// TwoSum), written from the method: it returns a pair (s, c) whose sum is the
// dot product with the accuracy of a float64 accumulation.
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace kvi {
namespace {

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

// Four independent Dot2 accumulations, one per float4 component, so that
// consecutive steps do not wait on each other; combined in a fixed order.
struct Dot2x4 {
    float s[4], c[4];
    __device__ __forceinline__ void zero()
    {
#pragma unroll
        for (int u = 0; u < 4; ++u) s[u] = c[u] = 0.f;
    }
    __device__ __forceinline__ void add(const float4 &q, const float4 &e)
    {
        dot2_step(q.x, e.x, s[0], c[0]);
        dot2_step(q.y, e.y, s[1], c[1]);
        dot2_step(q.z, e.z, s[2], c[2]);
        dot2_step(q.w, e.w, s[3], c[3]);
    }
    __device__ __forceinline__ void combine(float &so, float &co) const
    {
        float a, ea, b, eb;
        two_sum(s[0], s[1], a, ea);
        two_sum(s[2], s[3], b, eb);
        float t, et;
        two_sum(a, b, t, et);
        so = t;
        co = __fadd_rn(__fadd_rn(__fadd_rn(c[0], c[1]), __fadd_rn(c[2], c[3])),
                       __fadd_rn(__fadd_rn(ea, eb), et));
    }
};

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

// Selection key of a compensated score (s, c) without float64 arithmetic.
// TwoSum normalises the pair so that s' = fl(s' + c') and c' is the exact
// remainder.  Rounding to nearest is monotone, so for two scores the order of
// the exact values s' + c' is the lexicographic order of (s', c'); the key is
// the order-preserving images of s' (high word) and c' (low word).  -0 is
// folded onto +0 first.
__device__ __forceinline__ uint32_t order32(float x)
{
    const uint32_t u = __float_as_uint(__fadd_rn(x, 0.0f));
    return (u >> 31) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float unorder32(uint32_t o)
{
    return __uint_as_float((o >> 31) ? (o & 0x7fffffffu) : ~o);
}

__device__ __forceinline__ uint64_t score_key(float s, float c)
{
    float hi, lo;
    two_sum(s, c, hi, lo);
    return ((uint64_t)order32(hi) << 32) | order32(lo);
}

// The similarity reported for a key: s' = the score rounded to float32.
__device__ __forceinline__ float key_score(uint64_t key) { return unorder32((uint32_t)(key >> 32)); }

__device__ __forceinline__ bool better(uint64_t ka, int32_t ia, uint64_t kb, int32_t ib)
{
    return ka > kb || (ka == kb && ia < ib);
}

}  // namespace
}  // namespace kvi

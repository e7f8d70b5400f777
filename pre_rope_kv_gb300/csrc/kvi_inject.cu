// kvi_inject.cu -- gather, Chunked-RoPE rotate and paged scatter.
//
// "InferScale: GPU-Native KV Injection for Personalized LLM Serving":
// Section 5.1 / Theorem 6 (Chunked RoPE) -- each fact's keys are stored before
// rotary encoding and rotated to the positions they take in the prompt when
// injected; Section 3.4 -- K and V are scatter-copied into the engine's paged
// blocks before the forward pass, so only the query is prefilled.
//
// The kernel is a pure HBM stream: every injected byte is read once from the
// store and written once to the pool.  It is persistent (one CTA per SM,
// since the number of tokens is only known on the device in the fused path)
// and each CTA runs one deep bulk-copy pipeline:
//
//   - work is cut into pieces: up to `ct` consecutive tokens of one fact that
//     fall in one page (ct divides the page size), for one layer and one of
//     K/V, at most 8 KB; in the store and in the page a piece is one
//     contiguous run of bytes.  Items (piece, K|V, layer), layer innermost,
//     are handed out (fused calls) as one fixed first batch of 24 per CTA,
//     then in claims from a counter in the workspace that shrink as the work
//     runs out (guided self-scheduling), or (split calls) as one contiguous
//     range per CTA;
//   - small fused calls stage their requests' store views, block tables and
//     per-fact rows (written by the selector), positions and piece prefixes
//     in shared memory, so that resolving a piece takes no global round trip;
//   - a producer warp resolves 32 items at a time (one per lane) and each
//     lane moves its piece into its shared-memory stage (24 in all) with
//     cp.async.bulk, completion tracked by the stage's "full" mbarrier, so up
//     to 24 pieces (~170 KB) per SM are in flight whatever the registers
//     (issuing from all lanes: one issuing thread caps the copy rate);
//   - twelve consumer warps take the stages round-robin: a V piece is copied
//     out unchanged, a K piece is rotated (each lane takes rotate-half pairs
//     of one (token, vector) group, elements [8v, 8v+8) and
//     [D/2+8v, D/2+8v+8), for every head) and written with 16-byte stores;
//     the warp then releases the stage through its "empty" mbarrier.  A
//     consumer warp sees the same piece for several layers, so each lane
//     loads its cos/sin entries once per piece.
//
// Rotation accuracy.  The table holds cos and sin of p * omega_i computed in
// float64 on the host, split into a 16-significant-bit head and a float32
// tail.  A bf16 key has 8 significant bits, so x * head is exact in float32,
// and y = (x_i c_hi - x_j s_hi) + (x_i c_lo - x_j s_lo), whose first
// difference of exact products is rounded once, is within a few float32 ulps
// of the exact rotation at any position; one rounding to bf16 follows.
// Position 0 is the identity and copies the key bits.  The arithmetic runs
// on packed float32 pairs (two frequencies per instruction).
//
// Every wait is bounded (one second of globaltimer); a warp that times out
// records KVI_ERR_TIMEOUT and stops, and the warps waiting on it stop after
// their own bounded waits.  Before the producer warp exits it waits, again
// with a bound, for the last copy it issued into every stage, so no copy is
// still writing into the CTA's shared memory when the CTA ends.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "kvi_internal.cuh"
#include "kvi_sync.cuh"

namespace kvi {
namespace {

constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct PieceDesc {
    uint8_t *dst;
    uint32_t bytes;  // 0: nothing to do
    int32_t pos0;
    int32_t ntok;
    int16_t kv;
    int16_t stop;    // 1: no more pieces for this consumer
};

// Small fused calls (at most kCacheReqs requests, kCacheFacts fact slots and
// kCacheBlocks block-table entries) stage everything a piece's resolution
// needs in shared memory once per CTA, so that the producer resolves pieces
// without global round trips.
constexpr int kCacheReqs = 16;
constexpr int kCacheFacts = 272;   // R * (k + 1)
constexpr int kCacheBlocks = 1024; // R * max_blocks

struct ReqSlot {
    const void *kv;
    int64_t n_tokens;
    int32_t table_len;
    uint32_t flags;
};

struct FactSlot {
    int64_t row;  // the fact's first row in the store
    int32_t pos;  // its first position in the prompt
    int32_t len;  // its length (0: nothing to inject)
};

struct __align__(128) InjSmem {
    uint8_t stage[kInjRing][kPieceMax];
    uint64_t full[kInjRing];
    uint64_t empty[kInjRing];
    int32_t issued[kInjRing];  // last round whose "full" phase each stage started, -1: none
    PieceDesc desc[kInjRing];
    int32_t prefix[kMaxPrefix + 1];
    int32_t part[kInjThreads];
    ReqSlot req[kCacheReqs];
    FactSlot fact[kCacheFacts];
    int32_t fpc[kCacheFacts];
    int32_t btab[kCacheBlocks];
    // the pool's per-layer bases: each producer lane looks up its own layer,
    // which from the kernel parameters would be a divergent constant load
    uint8_t *lbase[KVI_MAX_LAYERS];
};
static_assert(sizeof(InjSmem) <= 227 * 1024, "inject shared memory");

// ------------------------------------------------------ async-copy helpers

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_u4(void *p, const uint4 &v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// --------------------------------------------------------------- rotation


__device__ __forceinline__ uint32_t pack_bf16(float a, float b)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half)
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Packed float32 pairs (Blackwell .f32x2 arithmetic): two adjacent
// frequencies are rotated by one instruction.  Each op rounds each half to
// nearest, exactly as the scalar op would.
__device__ __forceinline__ uint64_t f2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// bf16x2 (low half = first element) -> float32 pair
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t u)
{
    return f2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}
// float32 pair -> bf16x2, round to nearest even
__device__ __forceinline__ uint32_t f2_to_bf2(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return pack_bf16(lo, hi);
}

// Rotate 8 rotate-half pairs: lo holds x_i, hi holds x_{i+D/2}, for
// i = 8v .. 8v+7.  cs holds the table entries of those pairs, two pairs per
// 32 bytes: {cos_hi[i], cos_hi[i+1], cos_lo[i], cos_lo[i+1]},
// {sin_hi[i], sin_hi[i+1], sin_lo[i], sin_lo[i+1]}.  x * hi products are exact
// (8 x 16 significant bits), so y0 = x0 c - x1 s and y1 = x1 c + x0 s get one
// rounding of their main part plus a float32 tail correction.
// Rotate two pairs at once: x0 holds their first elements, x1 their second,
// c / sn the pairs' table entries.
__device__ __forceinline__ void rotate2(uint64_t x0, uint64_t x1, const float4 &c, const float4 &sn,
                                        uint64_t &y0, uint64_t &y1)
{
    const uint64_t chi = f2(c.x, c.y), clo = f2(c.z, c.w);
    const uint64_t shi = f2(sn.x, sn.y), slo = f2(sn.z, sn.w);
    y0 = add2(sub2(mul2(x0, chi), mul2(x1, shi)), sub2(mul2(x0, clo), mul2(x1, slo)));
    y1 = add2(add2(mul2(x1, chi), mul2(x0, shi)), add2(mul2(x1, clo), mul2(x0, slo)));
}

__device__ __forceinline__ void rotate8(uint4 &lo, uint4 &hi, const float4 *cs)
{
    uint32_t *pl = reinterpret_cast<uint32_t *>(&lo);
    uint32_t *ph = reinterpret_cast<uint32_t *>(&hi);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        uint64_t y0, y1;
        rotate2(bf2_to_f2(pl[w]), bf2_to_f2(ph[w]), cs[2 * w], cs[2 * w + 1], y0, y1);
        pl[w] = f2_to_bf2(y0);
        ph[w] = f2_to_bf2(y1);
    }
}

// Interleaved pairing: 16 consecutive elements a (8) then b (8) hold pairs
// (2i, 2i+1) for 8 consecutive i, one pair per 32-bit word.  The first and
// second elements of two adjacent pairs are gathered into float32 pairs,
// rotated as above and interleaved back.
__device__ __forceinline__ void rotate8_interleaved(uint4 &a, uint4 &b, const float4 *cs)
{
    uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t u = w[2 * g], v = w[2 * g + 1];
        const uint64_t x0 = f2(__uint_as_float(u << 16), __uint_as_float(v << 16));
        const uint64_t x1 = f2(__uint_as_float(u & 0xffff0000u), __uint_as_float(v & 0xffff0000u));
        uint64_t y0, y1;
        rotate2(x0, x1, cs[2 * g], cs[2 * g + 1], y0, y1);
        float y0a, y0b, y1a, y1b;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(y0a), "=f"(y0b) : "l"(y0));
        asm("mov.b64 {%0, %1}, %2;" : "=f"(y1a), "=f"(y1b) : "l"(y1));
        w[2 * g] = pack_bf16(y0a, y1a);
        w[2 * g + 1] = pack_bf16(y0b, y1b);
    }
    a = make_uint4(w[0], w[1], w[2], w[3]);
    b = make_uint4(w[4], w[5], w[6], w[7]);
}

// cos/sin entries of one (position, vector) pair group, kept in registers
// across the layers of a piece.
struct TableCache {
    int32_t p, v;
    float4 cs[8];
};

// Rotate a staged K piece ([ntok][hg][D] bf16) and write it to dst.  Lane
// c takes the (token, vector) group t = c / vph, v = c % vph -- pairs
// 8v .. 8v+7 -- loads their 8 cos/sin entries (cached across the layers of
// the piece) and walks the piece's heads.  Rotate-half: elements [8v, 8v+8)
// with [D/2+8v, D/2+8v+8); interleaved: elements [16v, 16v+16).  Lanes of
// one token cover contiguous bytes of a head, in shared memory and in the
// page.
__device__ __forceinline__ void rotate_piece(const InjectParams &p, const uint8_t *stg, uint8_t *dst,
                                             int ntok, int32_t pos0, int lane, TableCache &tc)
{
    const int D = p.D, HG = p.pg.hg, vph = D >> 4, half = D >> 1;
    const int groups = ntok * vph;
    for (int c = lane; c < groups; c += 32) {
        const int t = c / vph;
        const int v = c - t * vph;
        const int32_t pp = pos0 + t;
        if (pp != 0 && (pp != tc.p || v != tc.v)) {
            const float4 *tp = p.rope + (int64_t)pp * half + 8 * v;
#pragma unroll
            for (int e = 0; e < 8; ++e) tc.cs[e] = __ldg(tp + e);
            tc.p = pp;
            tc.v = v;
        }
        if (p.pairing == KVI_ROPE_PAIR_INTERLEAVED) {
            // group v: pairs 8v .. 8v+7 = elements 16v .. 16v+15
#pragma unroll 2
            for (int h = 0; h < HG; ++h) {
                const int off = ((t * HG + h) * D + 16 * v) * 2;
                uint4 a = *reinterpret_cast<const uint4 *>(stg + off);
                uint4 b = *reinterpret_cast<const uint4 *>(stg + off + 16);
                if (pp != 0) rotate8_interleaved(a, b, tc.cs);
                st_u4(dst + off, a);
                st_u4(dst + off + 16, b);
            }
            continue;
        }
#pragma unroll 2
        for (int h = 0; h < HG; ++h) {
            const int off = ((t * HG + h) * D + 8 * v) * 2;
            uint4 lo = *reinterpret_cast<const uint4 *>(stg + off);
            uint4 hi = *reinterpret_cast<const uint4 *>(stg + off + D);
            if (pp != 0) rotate8(lo, hi, tc.cs);
            st_u4(dst + off, lo);
            st_u4(dst + off + D, hi);
        }
    }
}

// Copy a staged V piece to dst, 16 bytes per lane per step.
__device__ __forceinline__ void copy_piece(const uint8_t *stg, uint8_t *dst, uint32_t bytes, int lane)
{
#pragma unroll 4
    for (uint32_t o = 16u * lane; o < bytes; o += 512u)
        st_u4(dst + o, *reinterpret_cast<const uint4 *>(stg + o));
}

// ----------------------------------------------------------------- pieces

// Largest j in [0, n) with a[j] <= x, for non-decreasing a[0..n] and
// a[0] <= x < a[n].
template <typename T, typename U>
__device__ __forceinline__ int search_le(const T *a, int n, U x)
{
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((U)a[mid] <= x) lo = mid;
        else hi = mid;
    }
    return lo;
}

struct Piece {
    const uint8_t *src;
    uint8_t *dst;
    uint32_t bytes;  // 0: nothing to do
    int32_t pos0;
    int32_t ntok;
    int32_t kv;
    bool direct;     // the store is in host memory: staged by cp.async, not a bulk copy
};

// What a piece needs to know about its fact and request.
struct FactRef {
    int32_t m;       // piece index within the fact
    int32_t len;     // fact length
    int64_t pos;     // fact's first position
    int64_t row;     // fact's first store row
    const void *kv;
    int64_t n_tokens;
    const int32_t *bt;  // block table (global or shared memory)
    int32_t tlen;
    uint32_t flags;     // the store's KVI_STORE_* flags
};

__device__ __forceinline__ FactRef fact_of_split(const InjectParams &p, const int32_t *prefix, int32_t piece)
{
    FactRef q;
    const int j = search_le(prefix, p.n, piece);
    q.m = piece - prefix[j];
    const int32_t f = p.ids[j];
    q.pos = p.pos[j];
    const kvi_store_view &sv = p.store.single;
    q.len = sv.fact_len[f];
    q.row = sv.fact_start[f];
    q.kv = sv.kv;
    q.n_tokens = sv.n_tokens;
    q.bt = p.block_tables;
    q.tlen = p.table_len;
    q.flags = sv.flags;
    return q;
}

// Request r's store: its own view, or the one store all requests share.
__device__ __forceinline__ const kvi_store_view &store_of(const InjectParams &p, int r)
{
    return p.store.many ? p.store.many[r] : p.store.single;
}

__device__ __forceinline__ FactRef fact_of_fused(const InjectParams &p, const int32_t *prefix, int32_t piece)
{
    FactRef q;
    const int r = search_le(prefix, p.R, piece);
    const int32_t local = piece - prefix[r];
    const int32_t *pcr = p.pc + (int64_t)r * (p.k + 1);
    const int j = search_le(pcr, p.k, local);
    q.m = local - pcr[j];
    q.pos = p.pos[(int64_t)r * p.k + j];
    q.len = p.slot_len[(int64_t)r * p.k + j];
    q.row = p.rows[(int64_t)r * p.k + j];
    const kvi_store_view &sv = store_of(p, r);
    q.kv = sv.kv;
    q.n_tokens = sv.n_tokens;
    q.bt = p.block_tables + (int64_t)r * p.max_blocks;
    q.tlen = p.table_lens[r];
    q.flags = sv.flags;
    return q;
}

__device__ __forceinline__ FactRef fact_of_cached(const InjectParams &p, const InjSmem &sm, int32_t piece)
{
    FactRef q;
    const int r = search_le(sm.prefix, p.R, piece);
    const int32_t local = piece - sm.prefix[r];
    const int32_t *pcr = sm.fpc + r * (p.k + 1);
    const int j = search_le(pcr, p.k, local);
    q.m = local - pcr[j];
    const FactSlot &fs = sm.fact[r * p.k + j];
    q.pos = fs.pos;
    q.len = fs.len;
    q.row = fs.row;
    const ReqSlot &rq = sm.req[r];
    q.kv = rq.kv;
    q.n_tokens = rq.n_tokens;
    q.bt = sm.btab + r * p.max_blocks;
    q.tlen = rq.table_len;
    q.flags = rq.flags;
    return q;
}

// Source, destination and extent of item `it` = (piece, K|V, layer), layer
// innermost; bytes = 0 (and the status set) when it falls outside the
// block table, the pool or the RoPE table.
__device__ __forceinline__ Piece resolve_piece(const InjectParams &p, const InjSmem &sm, bool cached,
                                               int64_t it)
{
    Piece x{nullptr, nullptr, 0u, 0, 0, 0, false};
    const int L2 = 2 * p.L;
    int64_t piece;
    int kl;
    if (it <= 0x7fffffff) {  // 32-bit division whenever the index allows it
        const uint32_t pu = (uint32_t)it / (uint32_t)L2;
        piece = pu;
        kl = (int)((uint32_t)it - pu * (uint32_t)L2);
    } else {
        piece = it / L2;
        kl = (int)(it - piece * L2);
    }
    const int kv = kl >= p.L ? 1 : 0;
    const int l = kl - kv * p.L;
    const FactRef q = cached ? fact_of_cached(p, sm, (int32_t)piece)
                      : p.fused ? fact_of_fused(p, sm.prefix, (int32_t)piece)
                                : fact_of_split(p, sm.prefix, (int32_t)piece);
    const int32_t mt = q.m / p.pg.units;
    const int32_t hg = q.m - mt * p.pg.units;
    // positions are non-negative int32 here: a fact that could be placed at
    // a negative or 64-bit position has no pieces
    const int64_t first = (uint32_t)q.pos / (uint32_t)p.pg.ct;
    const int64_t a = max(q.pos, (first + mt) * p.pg.ct);
    const int64_t b = min(q.pos + q.len, (first + mt + 1) * p.pg.ct);
    const int B = p.block_size;
    if (a < 0 || b <= a || b > (int64_t)q.tlen * B || b > p.rope_positions) {
        record_status(p.status, KVI_ERR_OUT_OF_RANGE);
        return x;
    }
    const uint32_t au = (uint32_t)a;  // 0 <= a < b <= rope_positions < 2^31
    const uint32_t page = au / (uint32_t)B;
    const int32_t blk = q.bt[page];
    if (blk < 0 || blk >= p.num_blocks) {
        record_status(p.status, KVI_ERR_OUT_OF_RANGE);
        return x;
    }
    const int64_t HD = (int64_t)p.H * p.D;
    const int64_t hoff = (int64_t)hg * p.pg.hg * p.D;
    const int64_t row = q.row + (a - q.pos);
    x.src = reinterpret_cast<const uint8_t *>(q.kv) +
            ((((int64_t)l * 2 + kv) * q.n_tokens + row) * HD + hoff) * 2;
    x.dst = sm.lbase[l] +
            ((((int64_t)kv * p.num_blocks + blk) * B + (au - page * (uint32_t)B)) * HD + hoff) * 2;
    x.ntok = (int32_t)(b - a);
    x.bytes = (uint32_t)(x.ntok * p.pg.hg * p.D * 2);
    x.pos0 = (int32_t)a;
    x.kv = kv;
    x.direct = (q.flags & KVI_STORE_KV_HOST) != 0;
    return x;
}

// counts in a[1..n] -> exclusive prefix a[0..n] (a[0] = 0), whole CTA.
__device__ void cta_prefix(int32_t *a, int n, int32_t *part)
{
    const int tid = threadIdx.x;
    const int per = (n + kInjThreads - 1) / kInjThreads;
    const int j0 = tid * per;
    int32_t run = 0;
    for (int j = j0; j < j0 + per && j < n; ++j) run += a[j + 1];
    part[tid] = run;
    __syncthreads();
    if (tid < 32) {
        int32_t carry = 0;
        for (int base = 0; base < kInjThreads; base += 32) {
            const int32_t v = part[base + tid];
            int32_t incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += t;
            }
            part[base + tid] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    __syncthreads();
    int32_t acc = part[tid];
    if (tid == 0) a[0] = 0;
    for (int j = j0; j < j0 + per && j < n; ++j) {
        acc += a[j + 1];
        a[j + 1] = acc;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kInjThreads, 1)
inject_kernel(const __grid_constant__ InjectParams p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    InjSmem &sm = *reinterpret_cast<InjSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid < kInjRing) {  // one stage's barriers per thread
        mbar_init(smem_u32(&sm.full[tid]), 1);
        mbar_init(smem_u32(&sm.empty[tid]), 1);
        sm.issued[tid] = -1;
        fence_async_smem();
    }
    for (int l = tid; l < p.L; l += kInjThreads) sm.lbase[l] = reinterpret_cast<uint8_t *>(p.layer_base[l]);

    // small fused calls: the requests' inputs (store views, block tables,
    // table lengths) are staged before the selection ends
    const bool cached = p.fused && p.R <= kCacheReqs && p.R * (p.k + 1) <= kCacheFacts &&
                        (int64_t)p.R * p.max_blocks <= kCacheBlocks;
    if (cached) {
        for (int i = tid; i < p.R * p.max_blocks; i += kInjThreads) sm.btab[i] = p.block_tables[i];
        for (int r = tid; r < p.R; r += kInjThreads) {
            const kvi_store_view &v = store_of(p, r);
            sm.req[r] = ReqSlot{v.kv, v.n_tokens, p.table_lens[r], v.flags};
        }
        __syncthreads();
    }

    pdl_wait();  // selection and placement of the previous kernel
    int count;
    if (p.fused) {
        count = p.R;
        for (int r = tid; r < p.R; r += kInjThreads) sm.prefix[r + 1] = p.npc[r];
        if (cached) {
            for (int e = tid; e < p.R * (p.k + 1); e += kInjThreads) sm.fpc[e] = p.pc[e];
            for (int e = tid; e < p.R * p.k; e += kInjThreads) {
                sm.fact[e] = FactSlot{p.rows[e], p.pos[e], p.slot_len[e]};
            }
        }
    } else {
        count = p.n;
        const kvi_store_view &st = p.store.single;
        for (int j = tid; j < p.n; j += kInjThreads) {
            const int32_t f = p.ids[j];
            const int64_t pos = p.pos[j];
            int32_t pieces = 0;
            if (f >= 0 && (int64_t)f < st.n_facts) {
                const int64_t s0 = st.fact_start[f];
                const int32_t l0 = st.fact_len[f];
                if (l0 >= 0 && s0 >= 0 && s0 + l0 <= st.n_tokens && pos >= 0) {
                    if (l0 > 0)
                        pieces = (int32_t)(((pos + l0 - 1) / p.pg.ct - pos / p.pg.ct + 1) * p.pg.units);
                } else {
                    record_status(p.status, KVI_ERR_OUT_OF_RANGE);
                }
            } else {
                record_status(p.status, KVI_ERR_OUT_OF_RANGE);
            }
            sm.prefix[j + 1] = pieces;
        }
    }
    if (tid == 0) sm.prefix[0] = 0;
    __syncthreads();
    if (count > 1) cta_prefix(sm.prefix, count, sm.part);  // one request: [0, npc] already
    const int64_t total = (int64_t)sm.prefix[count] * 2 * p.L;
    // static partition: a contiguous range of items per CTA (split calls);
    // dynamic (fused calls): CTA c first takes items [24c, 24c + 24), then
    // claims chunks of up to kInjRing items beyond the first 24 * grid from a
    // shared counter, which balances pieces of unequal size across SMs
    const bool dynamic = p.work != nullptr;
    const int64_t per = dynamic ? 0 : (total + gridDim.x - 1) / gridDim.x;
    const int64_t it0 = dynamic ? 0 : (int64_t)blockIdx.x * per;
    const int64_t n_static = total > it0 ? min(per, total - it0) : 0;
    const int64_t dyn0 = min(total, (int64_t)gridDim.x * kInjRing);

    if (warp == kInjConsumers) {
        // producer warp: each lane resolves one of kInjRing consecutive items
        // and issues its copy itself (a single issuing thread caps the
        // bulk-copy rate well below the SM's share of HBM bandwidth); each
        // lane waits on its own item's stage, and no two lanes of a batch
        // share one
        static_assert(kInjRing <= 32, "one batch per warp");
        int64_t local = 0;   // items this CTA has staged
        int64_t first;
        int nb;
        int want = kInjRing;        // size of the claim in flight
        unsigned long long claim = 0;  // lane 0: the claim in flight
        if (dynamic) {
            first = (int64_t)blockIdx.x * kInjRing;
            nb = (int)max((int64_t)0, min((int64_t)kInjRing, dyn0 - first));
            // the next claim goes out now; its latency overlaps this batch
            if (lane == 0) claim = atomicAdd(p.work, (unsigned long long)want);
        } else {
            first = it0;
            nb = (int)min((int64_t)kInjRing, n_static);
        }
        int64_t taken = nb;  // items of the static range taken
        bool ok = true;
        for (;;) {
            const int64_t j = local + lane;
            const int s = (int)(j % kInjRing);
            Piece x{nullptr, nullptr, 0u, 0, 0, 0, false};
            bool staged = false;  // this lane's stage is free and described
            if (lane < nb) {
                x = resolve_piece(p, sm, cached, first + lane);
                const int64_t round = j / kInjRing;
                if (round > 0 &&
                    !mbar_wait(smem_u32(&sm.empty[s]), (uint32_t)((round - 1) & 1), kWaitLimitNs)) {
                    record_status(p.status, KVI_ERR_TIMEOUT);
                    ok = false;
                } else {
                    staged = true;
                    sm.desc[s] = PieceDesc{x.dst, x.bytes, x.pos0, x.ntok, (int16_t)x.kv, 0};
                    sm.issued[s] = (int32_t)round;
                    const uint32_t fb = smem_u32(&sm.full[s]);
                    if (x.bytes && !x.direct) {
                        // the stage's previous contents were read by the
                        // consumers (generic proxy) before this async write
                        if (round > 0) fence_async_smem();
                        mbar_expect_tx(fb, x.bytes);
                        bulk_load(smem_u32(sm.stage[s]), x.src, x.bytes, fb);
                    } else if (!x.bytes) {
                        mbar_arrive(fb);
                    }
                }
            }
            // pieces of a host-resident store: the whole warp copies each
            // one into its stage with 16-byte cp.async (no bulk copy from
            // host memory); every lane's copies are tracked by the stage's
            // barrier, and one plain arrival completes its expected count
            uint32_t host = __ballot_sync(0xffffffffu, staged && x.bytes && x.direct);
            while (host) {
                const int i = __ffs(host) - 1;
                host &= host - 1;
                const uint8_t *src = reinterpret_cast<const uint8_t *>(
                    __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(x.src), i));
                const uint32_t bytes = __shfl_sync(0xffffffffu, x.bytes, i);
                const int si = __shfl_sync(0xffffffffu, s, i);
                const uint32_t dst = smem_u32(sm.stage[si]);
                for (uint32_t o = 16u * lane; o < bytes; o += 512u)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + o), "l"(src + o)
                                 : "memory");
                const uint32_t fb = smem_u32(&sm.full[si]);
                asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(fb) : "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(fb);
            }
            local += nb;
            if (!__all_sync(0xffffffffu, ok)) break;
            if (dynamic) {
                first = dyn0 + (int64_t)__shfl_sync(0xffffffffu, claim, 0);
                if (first >= total) break;
                nb = (int)min((int64_t)want, total - first);
                // guided self-scheduling: once fewer than two full claims per
                // CTA are left, claim a share of what is left (at least 2),
                // so that the CTAs run out of work at nearly the same time
                const int64_t left = total - first - nb;
                want = (int)max((int64_t)2, min((int64_t)kInjRing, left / (2 * (int64_t)gridDim.x)));
                if (lane == 0) claim = atomicAdd(p.work, (unsigned long long)want);
            } else {
                if (taken >= n_static) break;
                first = it0 + taken;
                nb = (int)min((int64_t)kInjRing, n_static - taken);
                taken += nb;
            }
        }
        // one stop descriptor for each consumer's next item
        if (ok && lane < kInjConsumers) {
            const int64_t j = local + lane;
            const int s = (int)(j % kInjRing);
            const int64_t round = j / kInjRing;
            if (round > 0 &&
                !mbar_wait(smem_u32(&sm.empty[s]), (uint32_t)((round - 1) & 1), kWaitLimitNs)) {
                record_status(p.status, KVI_ERR_TIMEOUT);
            } else {
                sm.desc[s] = PieceDesc{nullptr, 0u, 0, 0, 0, 1};
                sm.issued[s] = (int32_t)round;
                mbar_arrive(smem_u32(&sm.full[s]));
            }
        }
        // Leave no copy in flight into this CTA's shared memory: whatever
        // ended the loop (the last item, or a wait that gave up), the last
        // "full" phase the producer started on each stage (a copy, or a
        // plain arrival that completes at once) is waited for, with a
        // bound, before the producer exits.  The phase tracked must be the
        // last one: waiting on an earlier phase's parity after two more
        // phases began would wait on an incomplete phase of equal parity.
        __syncwarp();
        if (lane < kInjRing) {
            const int32_t r = sm.issued[lane];
            if (r >= 0 && !mbar_wait(smem_u32(&sm.full[lane]), (uint32_t)(r & 1), kWaitLimitNs))
                record_status(p.status, KVI_ERR_TIMEOUT);
        }
    } else {
        // consumers: this CTA's staged items warp, warp + 12, ... until a stop
        TableCache tc;
        tc.p = -1;
        tc.v = -1;
        for (int64_t j = warp;; j += kInjConsumers) {
            const int s = (int)(j % kInjRing);
            const uint32_t parity = (uint32_t)((j / kInjRing) & 1);
            const bool ok = mbar_wait(smem_u32(&sm.full[s]), parity, kWaitLimitNs);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) record_status(p.status, KVI_ERR_TIMEOUT);
                break;
            }
            const PieceDesc d = sm.desc[s];
            if (d.stop) break;
            const uint8_t *stg = sm.stage[s];
            if (d.bytes) {
                if (d.kv) copy_piece(stg, d.dst, d.bytes, lane);
                else rotate_piece(p, stg, d.dst, d.ntok, d.pos0, lane, tc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sm.empty[s]));
        }
    }
}

#ifdef KVI_DEBUG_CHECKS
// Debug builds: do two of the split call's facts target overlapping
// positions?  Fact j covers [pos[j], pos[j] + fact_len[ids[j]]) (facts with
// an invalid id or length are reported by the inject kernel itself); each
// thread compares its fact with every later one.
__global__ void __launch_bounds__(256) overlap_check_kernel(const __grid_constant__ InjectParams p)
{
    const kvi_store_view &st = p.store.single;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= p.n) return;
    auto extent = [&](int j, int64_t &a, int64_t &b) {
        const int32_t f = p.ids[j];
        a = b = 0;
        if (f < 0 || (int64_t)f >= st.n_facts) return;
        const int32_t len = st.fact_len[f];
        if (len <= 0) return;
        a = p.pos[j];
        b = a + len;
    };
    int64_t a0, b0;
    extent(i, a0, b0);
    if (b0 <= a0) return;
    for (int j = i + 1; j < p.n; ++j) {
        int64_t a1, b1;
        extent(j, a1, b1);
        if (b1 > a1 && a0 < b1 && a1 < b0) {
            record_status(p.status, KVI_ERR_INVALID_ARG);
            return;
        }
    }
}
#endif

}  // namespace

#ifdef KVI_DEBUG_CHECKS
cudaError_t launch_overlap_check(const InjectParams &p, cudaStream_t s)
{
    overlap_check_kernel<<<(unsigned)((p.n + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}
#endif

cudaError_t prepare_inject_kernel() { return smem_opt_in(inject_kernel, (int)sizeof(InjSmem)); }

cudaError_t launch_inject(const InjectParams &p, cudaStream_t s, bool pdl)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int smem = (int)sizeof(InjSmem);
    e = smem_opt_in(inject_kernel, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)di.sms);
    cfg.blockDim = dim3(kInjThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, inject_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace kvi

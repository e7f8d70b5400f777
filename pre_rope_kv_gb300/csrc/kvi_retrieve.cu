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
//   score_kernel   each warp streams a contiguous range of fact rows with the
//                  next row's 16-byte loads in flight while it reduces the
//                  current one; the query is re-read from L1.  The dot product
//                  is accumulated with Dot2 (Ogita, Rump & Oishi, "Accurate
//                  Sum and Dot Product", SIAM J. Sci. Comput. 26(6), 2005:
//                  error-free TwoProduct by FMA and TwoSum, carried as a
//                  float32 pair) and the pair becomes an exact 64-bit
//                  selection key with integer ordering only (no float64).
//                  The same warp validates the fact's extent in the store.
//   select_kernel  one CTA per request.  First a lower bound on the k-th
//                  key's top 16 bits is found from the best keys of 256
//                  disjoint key groups (one warp, binary search); the keys
//                  at or above it (usually little more than k) are ranked
//                  exactly.  When too many keys tie at that bound, a
//                  shared-memory histogram of the keys' float32 parts (a
//                  monotone map) finds the bucket that holds the k-th key;
//                  buckets above it are taken whole, the k-th bucket's keys
//                  are ranked exactly (or, when it is crowded, refined by an
//                  8-bit radix select on the full 64-bit key down to ties,
//                  which go to the lower fact id).
//                  In the fused path it also places the facts (rank order,
//                  back to back from the request's start) and cuts them into
//                  the inject kernel's pieces.
//   place_kernel   placement alone, for the split API.
#include <cuda_runtime.h>

#include "kvi_dot2.cuh"
#include "kvi_internal.cuh"

namespace kvi {
namespace {

// Bring `bytes` (a multiple of 16) at a 16-byte aligned address into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

constexpr int64_t kPrefetchRows = 8;

// First-level bucket (12 bits) of a key, from integer bit fields of s': its
// sign, its exponent clamped to [-48, 15] (6 bits) and the top 5 bits of its
// mantissa, i.e. 1/32-octave buckets for magnitudes 2^-48 .. 2^16 (coarser
// outside, where the clamp merges octaves).  Truncation and clamping never
// reverse an order, so key_a > key_b implies bucket_a >= bucket_b.
__device__ __forceinline__ uint32_t bucket_of(uint64_t key)
{
    const uint32_t o = (uint32_t)(key >> 32);
    const uint32_t u = (o >> 31) ? (o & 0x7fffffffu) : ~o;  // float bits of s'
    const int32_t e = (int32_t)((u >> 23) & 0xff) - 127 + 48;
    uint32_t mag;
    if (e < 0) mag = 0;
    else if (e > 63) mag = 2047;
    else mag = ((uint32_t)e << 5) | ((u >> 18) & 31u);
    return (u >> 31) ? 2047u - mag : 2048u + mag;
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

// Which request and fact a flat row index is, where its embedding starts
// (null when it is not a fact of a valid store), and its extent in the store
// (loaded with the row so that validating it costs no extra round trip).
struct RowRef {
    int32_t r;
    int64_t i;
    const float4 *e4;
    int64_t n_tokens;
    int64_t s0;
    int32_t l0;
};

struct ReqCache {
    int32_t r;
    bool ok;
    kvi_store_view st;
};

__device__ __forceinline__ RowRef resolve_row(const ScoreParams &p, int64_t g, ReqCache &rc,
                                              int lane)
{
    RowRef rr;
    rr.r = (int32_t)(g / p.max_facts);
    rr.i = g - (int64_t)rr.r * p.max_facts;
    if (rr.r != rc.r) {
        rc.r = rr.r;
        rc.st = load_store(p.store, rr.r);
        rc.ok = !p.store.many || store_ok(rc.st, p.g, p.max_facts, p.k);
    }
    const bool live = rc.ok && rr.i < rc.st.n_facts;
    rr.e4 = live ? reinterpret_cast<const float4 *>(rc.st.emb + rr.i * p.g.embed_dim) : nullptr;
    rr.n_tokens = rc.st.n_tokens;
    rr.s0 = 0;
    rr.l0 = -1;
    if (live && lane == 1) {
        rr.s0 = __ldg(rc.st.fact_start + rr.i);
        rr.l0 = __ldg(rc.st.fact_len + rr.i);
    }
    return rr;
}

// Key (lane 0) and validated length (lane 1) of one scored row.
__device__ __forceinline__ void finish_row(const ScoreParams &p, const RowRef &rr, float s,
                                           float c, int lane)
{
    warp_reduce_pair(s, c);
    const int64_t at = (int64_t)rr.r * p.key_stride + rr.i;
    if (lane == 0) p.keys[at] = score_key(s, c);
    if (lane == 1)
        p.lens[at] = (rr.l0 >= 0 && rr.s0 >= 0 && rr.s0 + rr.l0 <= rr.n_tokens) ? rr.l0 : -1;
}

template <int NV>  // float4 per lane per row (E = 128 * NV); 0 = any E % 4 == 0
__global__ void __launch_bounds__(kScoreThreads, 2)
score_kernel(const __grid_constant__ ScoreParams p)
{
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t G = (int64_t)gridDim.x * (kScoreThreads / 32);
    const int64_t gw = (int64_t)blockIdx.x * (kScoreThreads / 32) + (threadIdx.x >> 5);
    const int64_t total = (int64_t)p.R * p.max_facts;
    const int64_t per = (total + G - 1) / G;
    const int64_t g0 = gw * per;
    const int64_t g1 = min(total, g0 + per);
    if (g0 >= g1) return;
    const int E = p.g.embed_dim;

    ReqCache rc;
    rc.r = -1;
    rc.ok = false;
    // keep the next kPrefetchRows rows of this warp's range on their way into
    // L2 (bulk prefetch, no registers), so that each row's loads hit L2; rows
    // of another request than the cached one are left to the plain loads
    const int64_t row_bytes = (int64_t)E * 4;
    int64_t pf = g0;
    auto prefetch_to = [&](int64_t upto) {
        upto = min(upto, g1);
        while (pf < upto) {
            const int32_t r = (int32_t)(pf / p.max_facts);
            const int64_t i = pf - (int64_t)r * p.max_facts;
            const int64_t seg = min(upto, (int64_t)(r + 1) * p.max_facts) - pf;
            if (lane == 0 && r == rc.r && rc.ok) {
                const int64_t n = min(seg, rc.st.n_facts - i);
                if (n > 0) bulk_prefetch_l2(rc.st.emb + i * E, (uint32_t)(n * row_bytes));
            }
            pf += seg;
        }
    };
    if constexpr (NV > 0) {
        // double-buffered rows where registers allow it (E <= 1024)
        // the query is read per row from L1 (it stays resident there)
        constexpr bool kDB = NV <= 8;
        float4 cur[NV], nxt[kDB ? NV : 1];
        RowRef a = resolve_row(p, g0, rc, lane);
        prefetch_to(g0 + 1 + kPrefetchRows);
        if (a.e4) {
#pragma unroll
            for (int m = 0; m < NV; ++m) cur[m] = ld_stream_f4(a.e4 + lane + 32 * m);
        }
        for (int64_t g = g0; g < g1; ++g) {
            prefetch_to(g + 1 + kPrefetchRows);
            RowRef b{0, 0, nullptr, 0, 0, -1};
            if (kDB && g + 1 < g1) {
                b = resolve_row(p, g + 1, rc, lane);
                if (b.e4) {
#pragma unroll
                    for (int m = 0; m < (kDB ? NV : 1); ++m) nxt[m] = ld_stream_f4(b.e4 + lane + 32 * m);
                }
            }
            if (a.e4) {
                const float4 *q4 = reinterpret_cast<const float4 *>(p.queries + (int64_t)a.r * E);
                float s = 0.f, c = 0.f;
#pragma unroll
                for (int m = 0; m < NV; ++m) dot2_f4(__ldg(q4 + lane + 32 * m), cur[m], s, c);
                finish_row(p, a, s, c, lane);
            }
            if constexpr (kDB) {
                a = b;
#pragma unroll
                for (int m = 0; m < NV; ++m) cur[m] = nxt[m];
            } else if (g + 1 < g1) {
                a = resolve_row(p, g + 1, rc, lane);
                if (a.e4) {
#pragma unroll
                    for (int m = 0; m < NV; ++m) cur[m] = ld_stream_f4(a.e4 + lane + 32 * m);
                }
            }
        }
    } else {
        for (int64_t g = g0; g < g1; ++g) {
            const RowRef a = resolve_row(p, g, rc, lane);
            prefetch_to(g + 1 + kPrefetchRows);
            if (!a.e4) continue;
            const float4 *q4 = reinterpret_cast<const float4 *>(p.queries + (int64_t)a.r * E);
            float s = 0.f, c = 0.f;
            for (int v = lane; v < E / 4; v += 32) dot2_f4(__ldg(q4 + v), ld_stream_f4(a.e4 + v), s, c);
            finish_row(p, a, s, c, lane);
        }
    }
}

// Ring variant (rows of at most 8 KB, i.e. E <= 2048): one CTA per SM; a
// producer warp (all lanes issuing) streams the CTA's contiguous range of
// fact rows into a ring
// of shared-memory stages (one row per stage, 192 KB in all) with
// cp.async.bulk, and 24 consumer warps take the rows round-robin, each lane
// reading its float4 slots from shared memory and keeping four independent
// Dot2 accumulators.  The Dot2 arithmetic (about ten float32 operations per
// element) is what limits the rate at which an SM retires rows, so the
// consumers are as many warps as the registers allow (24 measured 1.2 us
// faster than 12 on a 10k-fact store).  The extents of a warp's next 32 rows are
// fetched together (one per lane), so validating them costs one round trip
// per 32 rows.  The code is kept short: it is fetched cold on every launch.

constexpr int kRingConsumers = 24;
constexpr int kRingThreads = (kRingConsumers + 1) * 32;
constexpr int kRingBytes = 192 * 1024;
constexpr int kRingMaxStages = 96;
constexpr uint64_t kRingWaitNs = 1000000000ull;

struct ScoreRingSmem {
    uint8_t ring[kRingBytes];
    uint64_t full[kRingMaxStages];
    uint64_t empty[kRingMaxStages];
    int32_t issued[kRingMaxStages];  // last round whose "full" phase each stage started, -1: none
};

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __noinline__ bool ring_wait(uint32_t bar, uint32_t parity)
{
    uint64_t t0 = 0;
    for (int it = 0;; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            "selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (it == 0) t0 = t;
        else if (t - t0 > kRingWaitNs) return false;
    }
}

// Flat row g of the R x max_facts row space, advanced without divisions.
struct RowCursor {
    int32_t r;
    int64_t i;
    __device__ void init(int64_t g, int64_t max_facts)
    {
        r = (int32_t)(g / max_facts);
        i = g - (int64_t)r * max_facts;
    }
    __device__ void advance(int64_t by, int64_t max_facts)
    {
        i += by;
        while (i >= max_facts) {
            i -= max_facts;
            ++r;
        }
    }
};

#ifdef KVI_DEBUG_CHECKS
// Debug builds: flat row whose copy the scoring kernel skips (negative: none),
// set by kvi_debug_stall_scorer_row to make a bounded wait run out.
__device__ long long g_debug_stall_row = -1;
#endif

struct StoreCache {
    int32_t r;
    bool ok;
    kvi_store_view st;
    __device__ void get(const ScoreParams &p, int32_t rr)
    {
        if (rr == r) return;
        r = rr;
        st = load_store(p.store, rr);
        ok = !p.store.many || store_ok(st, p.g, p.max_facts, p.k);
    }
    __device__ bool live(int64_t i) const { return ok && i < st.n_facts; }
};

__global__ void __launch_bounds__(kRingThreads, 1)
score_ring_kernel(const __grid_constant__ ScoreParams p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    ScoreRingSmem &sm = *reinterpret_cast<ScoreRingSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.g.embed_dim;
    const uint32_t row_bytes = (uint32_t)E * 4u;
    const int S = min(kRingMaxStages, (int)(kRingBytes / row_bytes));
    if (tid < S) {  // one stage's barriers per thread
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.full[tid])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.empty[tid])) : "memory");
        sm.issued[tid] = -1;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    const int64_t total = (int64_t)p.R * p.max_facts;
    const int64_t per = (total + gridDim.x - 1) / gridDim.x;
    const int64_t g0 = (int64_t)blockIdx.x * per;
    const int64_t n = total > g0 ? min(per, total - g0) : 0;  // rows of this CTA
    // the store view of this CTA's first request is loaded while the
    // barriers are set up
    StoreCache sc;
    sc.r = -1;
    sc.ok = false;
    if (n > 0) sc.get(p, (int32_t)(g0 / p.max_facts));
    __syncthreads();
    pdl_launch_dependents();

    if (warp == kRingConsumers) {
        // producer warp: every lane issues copies, rows base + lane for
        // base = 0, 32, 64, ... (a single issuing thread caps the bulk-copy
        // rate far below the SM's share of HBM bandwidth); each lane waits on
        // its own row's stage
        for (int64_t base = 0; base < n; base += 32) {
            const int64_t j = base + lane;
            bool ok = true;
            if (j < n) {
                const int s = (int)(j % S);
                const uint32_t round = (uint32_t)(j / S);
                RowCursor cur;
                cur.init(g0 + j, p.max_facts);
                if (round > 0 && !ring_wait(smem_addr(&sm.empty[s]), (round - 1) & 1u)) {
                    record_status(p.status, KVI_ERR_TIMEOUT);
                    ok = false;
                } else {
                    sc.get(p, cur.r);
                    const uint32_t fb = smem_addr(&sm.full[s]);
#ifdef KVI_DEBUG_CHECKS
                    // no copy and no arrival for this row: its consumer's
                    // wait runs out
                    const bool stall = g0 + j == g_debug_stall_row;
#else
                    constexpr bool stall = false;
#endif
                    if (stall) {
                    } else if (sc.live(cur.i)) {
                        sm.issued[s] = (int32_t)round;
                        if (round > 0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fb),
                                     "r"(row_bytes)
                                     : "memory");
                        asm volatile(
                            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], "
                            "%2, [%3];" ::"r"(smem_addr(sm.ring + (size_t)s * row_bytes)),
                            "l"(sc.st.emb + cur.i * E), "r"(row_bytes), "r"(fb)
                            : "memory");
                    } else {
                        sm.issued[s] = (int32_t)round;
                        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(fb) : "memory");
                    }
                }
            }
            if (!__all_sync(0xffffffffu, ok)) break;
        }
        // no copy may still be writing into shared memory when the CTA
        // ends: wait (bounded) for the last "full" phase started on every
        // stage (a copy, or an arrival that completes at once), whether the
        // loop finished or a wait gave up
        __syncwarp();
        for (int s = lane; s < S; s += 32) {
            const int32_t r = sm.issued[s];
            if (r >= 0 && !ring_wait(smem_addr(&sm.full[s]), (uint32_t)r & 1u))
                record_status(p.status, KVI_ERR_TIMEOUT);
        }
        return;
    }

    // consumers: rows warp, warp + 12, ...  The extents of the next 32 of a
    // warp's rows are loaded together, one per lane, and handed to the row's
    // finishing lanes with shuffles, so their latency is paid once per 32 rows.
    RowCursor cur;
    cur.init(g0 + warp, p.max_facts);
    int s = warp % S;
    uint32_t round = (uint32_t)(warp / S);
    int64_t bs0 = 0;
    int32_t bl0 = -1;
#pragma unroll 1
    for (int64_t j = warp, m = 0; j < n; j += kRingConsumers, ++m) {
        if ((m & 31) == 0) {
            // lane l: extent of this warp's row j + 12 l
            RowCursor c = cur;
            c.advance((int64_t)lane * kRingConsumers, p.max_facts);
            bs0 = 0;
            bl0 = -1;
            if (j + (int64_t)lane * kRingConsumers < n) {
                sc.get(p, c.r);
                if (sc.live(c.i)) {
                    bs0 = __ldg(sc.st.fact_start + c.i);
                    bl0 = __ldg(sc.st.fact_len + c.i);
                }
            }
        }
        const int64_t s0 = __shfl_sync(0xffffffffu, bs0, (int)(m & 31));
        const int32_t l0 = __shfl_sync(0xffffffffu, bl0, (int)(m & 31));
        const bool ok = ring_wait(smem_addr(&sm.full[s]), round & 1u);
        if (!__all_sync(0xffffffffu, ok)) {
            if (lane == 0) record_status(p.status, KVI_ERR_TIMEOUT);
            // the rows this warp will not score keep stale keys and lengths
            // in the workspace: mark their lengths invalid, so that a fused
            // call injects nothing from them (placement reports them)
            for (int64_t jj = j + (int64_t)lane * kRingConsumers; jj < n; jj += 32 * (int64_t)kRingConsumers) {
                RowCursor c;
                c.init(g0 + jj, p.max_facts);
                p.lens[(int64_t)c.r * p.key_stride + c.i] = -1;
            }
            return;
        }
        sc.get(p, cur.r);
        if (sc.live(cur.i)) {
            const float4 *row = reinterpret_cast<const float4 *>(sm.ring + (size_t)s * row_bytes);
            const float4 *q4 = reinterpret_cast<const float4 *>(p.queries + (int64_t)cur.r * E);
            Dot2x4 acc;
            acc.zero();
#pragma unroll 4
            for (int v = lane; v < E / 4; v += 32) acc.add(__ldg(q4 + v), row[v]);
            float sacc, cacc;
            acc.combine(sacc, cacc);
            RowRef rr;
            rr.r = cur.r;
            rr.i = cur.i;
            rr.e4 = nullptr;
            rr.n_tokens = sc.st.n_tokens;
            rr.s0 = s0;
            rr.l0 = l0;
            finish_row(p, rr, sacc, cacc, lane);
        }
        __syncwarp();
        if (lane == 0)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&sm.empty[s])) : "memory");
        cur.advance(kRingConsumers, p.max_facts);
        s += kRingConsumers;
        while (s >= S) {
            s -= S;
            ++round;
        }
    }
}

// ---------------------------------------------------------------- selection

// Inclusive scan of one value per thread over a 1024-thread block.
template <typename T>
__device__ __forceinline__ T block_incl_scan(T v, T *warp_tot)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const T t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    if (warp == 0) {
        T w = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const T t = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += t;
        }
        warp_tot[lane] = w;
    }
    __syncthreads();
    const T before = warp ? warp_tot[warp - 1] : T(0);
    __syncthreads();  // warp_tot is reused by the next call
    return v + before;
}

struct SelectSmem {
    uint32_t hist[kHistBins];
    uint64_t cand_key[kCandCap];
    int32_t cand_id[kCandCap];
    int32_t cand_len[kCandCap];
    uint64_t sure_key[KVI_MAX_K];
    int32_t sure_id[KVI_MAX_K];
    int32_t sure_len[KVI_MAX_K];
    uint64_t out_key[KVI_MAX_K];
    int32_t out_id[KVI_MAX_K];
    int32_t out_len[KVI_MAX_K];
    int32_t out_pc[KVI_MAX_K];
    uint32_t warp_tot[32];
    int64_t out_s0[KVI_MAX_K];  // placement: first store row of each selected fact
    int64_t wsum[32];   // placement: lengths per warp
    int32_t wpc[32];    // placement: inject pieces per warp
    uint32_t n_sure, n_cand, bucket, above, digit, above2, pop;
};

// Rank of entry e among n entries (keys[], ids[]): how many of them are
// better.  One warp per entry, the lanes splitting the comparisons.
__device__ __forceinline__ uint32_t warp_rank(const uint64_t *keys, const int32_t *ids, uint32_t n,
                                              uint64_t ke, int32_t ie, int lane)
{
    uint32_t rank = 0;
    for (uint32_t o = lane; o < n; o += 32) rank += better(keys[o], ids[o], ke, ie);
    return __reduce_add_sync(0xffffffffu, rank);
}

// Rank the n_cand candidates in shared memory and move the best `need` of
// them to the sure list (positions base .. base + need).
__device__ void take_best_candidates(SelectSmem &sm, uint32_t n_cand, uint32_t need, uint32_t base)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (uint32_t c = warp; c < n_cand; c += kSelectThreads / 32) {
        const uint64_t kc = sm.cand_key[c];
        const int32_t ic = sm.cand_id[c];
        const uint32_t rank = warp_rank(sm.cand_key, sm.cand_id, n_cand, kc, ic, lane);
        if (lane == 0 && rank < need && base + rank < (uint32_t)KVI_MAX_K) {
            sm.sure_key[base + rank] = kc;
            sm.sure_id[base + rank] = ic;
            sm.sure_len[base + rank] = sm.cand_len[c];
        }
    }
}

__device__ __forceinline__ void add_sure(SelectSmem &sm, uint64_t key, int32_t id, int32_t len)
{
    const uint32_t at = atomicAdd(&sm.n_sure, 1u);
    if (at < (uint32_t)KVI_MAX_K) {
        sm.sure_key[at] = key;
        sm.sure_id[at] = id;
        sm.sure_len[at] = len;
    }
}

__device__ __forceinline__ void add_cand(SelectSmem &sm, uint64_t key, int32_t id, int32_t len)
{
    const uint32_t at = atomicAdd(&sm.n_cand, 1u);
    if (at < (uint32_t)kCandCap) {
        sm.cand_key[at] = key;
        sm.cand_id[at] = id;
        sm.cand_len[at] = len;
    }
}

// Radix refinement of a crowded first-level bucket b0 on the full 64-bit
// keys (read from global memory), down to ties broken by the lower id.  Kept
// out of line: it is rarely taken and its code need not be fetched otherwise.
__device__ __noinline__ void select_crowded(SelectSmem &sm, const uint64_t *keys, const int32_t *lens,
                               int64_t N, uint32_t b0, uint32_t need)
{
    const int tid = threadIdx.x;
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
        for (int64_t i = tid; i < N; i += kSelectThreads) {
            const uint64_t key = __ldcg(keys + i);
            if (bucket_of(key) != b0) continue;
            if (shift < 56 && (key >> (shift + 8)) != prefix) continue;
            if (((key >> shift) & 0xff) > dd) add_sure(sm, key, (int32_t)i, __ldcg(lens + i));
        }
        need_r -= above2;
        prefix = (prefix << 8) | dd;
        if (tid == 0) sm.n_cand = 0;
        __syncthreads();
        if (M2 <= (uint32_t)kCandCap) {
            for (int64_t i = tid; i < N; i += kSelectThreads) {
                const uint64_t key = __ldcg(keys + i);
                if (bucket_of(key) == b0 && (key >> shift) == prefix)
                    add_cand(sm, key, (int32_t)i, __ldcg(lens + i));
            }
            __syncthreads();
            take_best_candidates(sm, M2, need_r, sm.n_sure);
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
            const uint32_t incl = block_incl_scan<uint32_t>(flag, sm.warp_tot);
            const uint32_t at = taken + incl - flag;
            if (flag && at < need_r && base + at < (uint32_t)KVI_MAX_K) {
                sm.sure_key[base + at] = key;
                sm.sure_id[base + at] = (int32_t)i;
                sm.sure_len[base + at] = __ldcg(lens + i);
            }
            taken += sm.warp_tot[31];  // block total of the flags
            __syncthreads();
        }
    }
    __syncthreads();
}

// Selection by histogram (the general path): a shared-memory histogram of
// the keys' float32 parts finds the bucket that holds the k-th key; buckets
// above it are taken whole and the k-th bucket's keys are ranked exactly or,
// when it is crowded, refined by radix selection.  Keys stream from L2.  On
// return sm.out_* hold the k best in rank order.  Kept out of line: it runs
// only when many keys tie, and the common path's code stays contiguous.
__device__ __noinline__ void select_by_histogram(SelectSmem &sm, const uint64_t *keys,
                                                 const int32_t *lens, int64_t N, int32_t k)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // 1. histogram of the first-level buckets (hist is zero on entry)
#pragma unroll 4
    for (int64_t i = tid; i < N; i += kSelectThreads) atomicAdd(&sm.hist[bucket_of(__ldcg(keys + i))], 1u);
    __syncthreads();
    // 2. the bucket holding the k-th key (bucket 4095 is the best);
    //    thread t owns buckets 4095-4t .. 4092-4t.
    const int top = kHistBins - 1 - 4 * tid;
    const uint32_t c0 = sm.hist[top], c1 = sm.hist[top - 1];
    const uint32_t c2 = sm.hist[top - 2], c3 = sm.hist[top - 3];
    const uint32_t incl = block_incl_scan<uint32_t>(c0 + c1 + c2 + c3, sm.warp_tot);
    const uint32_t excl = incl - (c0 + c1 + c2 + c3);
    if (excl < (uint32_t)k && incl >= (uint32_t)k) {
        const uint32_t cs[4] = {c0, c1, c2, c3};
        uint32_t run = excl;
        for (int j = 0; j < 4; ++j) {
            if (run + cs[j] >= (uint32_t)k) {
                sm.bucket = (uint32_t)(top - j);
                sm.above = run;
                sm.pop = cs[j];
                break;
            }
            run += cs[j];
        }
    }
    __syncthreads();
    const uint32_t b0 = sm.bucket;
    const uint32_t above = sm.above;
    const uint32_t M = sm.pop;
    const uint32_t need = (uint32_t)k - above;

    // 3. keys above the bucket are in; keys in it are candidates.
    const bool direct = M <= (uint32_t)kCandCap;
#pragma unroll 4
    for (int64_t i = tid; i < N; i += kSelectThreads) {
        const uint64_t key = __ldcg(keys + i);
        const uint32_t b = bucket_of(key);
        if (b > b0) add_sure(sm, key, (int32_t)i, __ldcg(lens + i));
        else if (b == b0 && direct) add_cand(sm, key, (int32_t)i, __ldcg(lens + i));
    }
    __syncthreads();
    if (direct) {
        // 4. the k selected keys in rank order, in one pass: every key above
        //    the bucket is better than every key in it, so the former are
        //    ranked among themselves (ranks 0 .. above-1) and the bucket's
        //    keys among themselves (from rank `above`)
        for (uint32_t e = warp; e < above + M; e += kSelectThreads / 32) {
            if (e < above) {
                const uint64_t ke = sm.sure_key[e];
                const int32_t ie = sm.sure_id[e];
                const uint32_t rank = warp_rank(sm.sure_key, sm.sure_id, above, ke, ie, lane);
                if (lane == 0 && rank < above) {
                    sm.out_key[rank] = ke;
                    sm.out_id[rank] = ie;
                    sm.out_len[rank] = sm.sure_len[e];
                }
            } else {
                const uint32_t c = e - above;
                const uint64_t kc = sm.cand_key[c];
                const int32_t ic = sm.cand_id[c];
                const uint32_t rank = warp_rank(sm.cand_key, sm.cand_id, M, kc, ic, lane);
                if (lane == 0 && rank < need) {
                    sm.out_key[above + rank] = kc;
                    sm.out_id[above + rank] = ic;
                    sm.out_len[above + rank] = sm.cand_len[c];
                }
            }
        }
    } else {
        select_crowded(sm, keys, lens, N, b0, need);
        __syncthreads();
        // 4. the k selected keys in rank order.
        for (int e = warp; e < k; e += kSelectThreads / 32) {
            const uint64_t ke = sm.sure_key[e];
            const int32_t ie = sm.sure_id[e];
            const uint32_t rank = warp_rank(sm.sure_key, sm.sure_id, (uint32_t)k, ke, ie, lane);
            if (lane == 0 && rank < (uint32_t)KVI_MAX_K) {
                sm.out_key[rank] = ke;
                sm.out_id[rank] = ie;
                sm.out_len[rank] = sm.sure_len[e];
            }
        }
    }
    __syncthreads();
}

// Keys a selecting CTA can keep (16 bits each) in shared memory past
// SelectSmem: stores of up to this many facts (or candidates) are read from
// L2 once.
constexpr int64_t kSmemKeysMax = 65536;
static_assert(sizeof(SelectSmem) + 2 * kSmemKeysMax <= 227 * 1024, "select smem");

constexpr int kWarmFacts = 8;
constexpr int kStreamUnroll = 8;  // key loads in flight per thread when staging to shared memory
constexpr int kSelectGroups = 256;

// t* = the largest t such that at least k of the 256 values v (8 per lane of
// the calling warp) are >= t, for 1 <= k <= 256.  The smallest value always
// qualifies and max + 1 never does, so a 4-ary search between the two
// (three independent warp counts per round) finds t* in log4 of the range
// of values rounds.
__device__ __forceinline__ uint32_t kth_largest_bound(const uint32_t (&v)[kSelectGroups / 32], uint32_t k)
{
    uint32_t vmin = v[0], vmax = v[0];
#pragma unroll
    for (int i = 1; i < kSelectGroups / 32; ++i) {
        vmin = min(vmin, v[i]);
        vmax = max(vmax, v[i]);
    }
    uint32_t lo = __reduce_min_sync(0xffffffffu, vmin);
    uint32_t hi = __reduce_max_sync(0xffffffffu, vmax) + 1u;
    while (hi - lo > 1) {
        const uint32_t d = hi - lo;
        const uint32_t m1 = lo + d / 4, m2 = lo + d / 2, m3 = lo + (3 * d) / 4;
        uint32_t a1 = 0, a2 = 0, a3 = 0;
#pragma unroll
        for (int i = 0; i < kSelectGroups / 32; ++i) {
            a1 += v[i] >= m1 ? 1u : 0u;
            a2 += v[i] >= m2 ? 1u : 0u;
            a3 += v[i] >= m3 ? 1u : 0u;
        }
        const uint32_t c1 = __reduce_add_sync(0xffffffffu, a1);
        const uint32_t c2 = __reduce_add_sync(0xffffffffu, a2);
        const uint32_t c3 = __reduce_add_sync(0xffffffffu, a3);
        // count(>= lo) >= k > count(>= hi) stays true; equal midpoints
        // give equal counts, so each branch shrinks the range
        if (c3 >= k) lo = m3;
        else if (c2 >= k) { lo = m2; hi = m3; }
        else if (c1 >= k) { lo = m1; hi = m2; }
        else hi = m1;
    }
    return lo;
}

// Placement of one request (Figure 2 caption, "positioned by chunked RoPE";
// rank order, back to back from the request's start), one thread per
// selected fact j < k: its length, the exclusive prefix of the lengths (its
// position) and of its inject pieces, by warp scans and one table of warp
// totals.  Also writes each fact's first store row for the inject kernel
// (so that it needs no dependent load of fact_start) and, from the spare
// warps, touches the first facts it will move -- every layer's K and V rows
// of the best-ranked kWarmFacts facts, which the inject kernel's first items
// cover -- with one 128-byte L2 prefetch each, which warms their address
// translations (device-resident stores only; prefetching whole runs from one
// SM is far too slow: its bulk-copy unit moves them one after another).  All
// threads of the CTA call this.
__device__ __forceinline__ void place_parallel(const SelectParams &p, SelectSmem &sm, int r, bool ok,
                                               const kvi_store_view &st, int64_t start, int32_t tl)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t k = p.k;
    const int kw = (k + 31) / 32;  // warps holding a fact
    const int j = tid;
    int32_t len = 0;
    int32_t f = -1;
    int64_t s0 = 0;
    if (j < k && ok) {
        f = sm.out_id[j];
        len = sm.out_len[j];
        if (f < 0 || (int64_t)f >= st.n_facts || len < 0) {
            record_status(p.status, KVI_ERR_OUT_OF_RANGE);
            len = 0;
        }
        // lengths are -1 unless the scoring kernel found the extent inside
        // the store; only facts with a row inject anything
        if (len > 0) s0 = __ldg(st.fact_start + f);
    }
    if (!ok && tid == 0) record_status(p.status, KVI_ERR_OUT_OF_RANGE);
    int64_t incl = len;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (warp < kw && lane == 31) sm.wsum[warp] = incl;
    __syncthreads();
    int64_t before = 0, total = 0;
    for (int w = 0; w < kw; ++w) {
        const int64_t t = sm.wsum[w];
        before += w < warp ? t : 0;
        total += t;
    }
    int fit = ok ? 1 : 0;
    if (tl < 0 || tl > p.max_blocks) {
        if (tid == 0) record_status(p.status, KVI_ERR_OUT_OF_RANGE);
        fit = 0;
    } else if (start < 0 || start + total > (int64_t)tl * p.block_size) {
        if (tid == 0 && ok) record_status(p.status, KVI_ERR_CAPACITY);
        fit = 0;
    }
    const int64_t run = start + before + incl - len;  // this fact's first position
    int32_t pc = 0;
    if (j < k) {
        if (fit && len > 0) {  // positions fit 31 bits once the request fits its table
            const uint32_t ct = (uint32_t)p.pg.ct;
            const uint32_t first = (uint32_t)run / ct, last = (uint32_t)(run + len - 1) / ct;
            pc = (int32_t)((last - first + 1) * (uint32_t)p.pg.units);
        }
        p.pos[(int64_t)r * k + j] = (int32_t)run;
        p.slot_len[(int64_t)r * k + j] = len;
        if (ok) p.rows[(int64_t)r * k + j] = s0;
        sm.out_s0[j] = s0;
    }
    int32_t pin = pc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xffffffffu, pin, o);
        if (lane >= o) pin += t;
    }
    if (warp < kw && lane == 31) sm.wpc[warp] = pin;
    __syncthreads();
    int32_t pbefore = 0, ptotal = 0;
    for (int w = 0; w < kw; ++w) {
        const int32_t t = sm.wpc[w];
        pbefore += w < warp ? t : 0;
        ptotal += t;
    }
    if (j < k) p.pc[(int64_t)r * (k + 1) + j] = pbefore + pin - pc;
    if (tid == 0) {
        p.pc[(int64_t)r * (k + 1) + k] = ptotal;
        p.npc[r] = ptotal;
    }
    // warm the first facts' translations (warps past the ones holding
    // facts; the rows were stored in shared memory before the last barrier)
    if (ok && warp >= kw && !(st.flags & KVI_STORE_KV_HOST)) {
        const int L = p.g.layers;
        const int64_t row_bytes = (int64_t)p.g.kv_heads * p.g.head_dim * 2;
        const int nf = min(k, kWarmFacts);
        for (int e = tid - 32 * kw; e < nf * 2 * L; e += kSelectThreads - 32 * kw) {
            const int jj = e / (2 * L);
            const int plane = e - jj * 2 * L;  // layer * 2 + (K|V)
            const int32_t ln = sm.out_len[jj];
            const int64_t a0 = sm.out_s0[jj];
            if (ln <= 0 || a0 < 0 || a0 + ln > st.n_tokens) continue;
            const uint8_t *src = reinterpret_cast<const uint8_t *>(st.kv) +
                                 ((int64_t)plane * st.n_tokens + a0) * row_bytes;
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], 128;" ::"l"(src) : "memory");
        }
    }
}

__global__ void __launch_bounds__(kSelectThreads, 1)
select_kernel(const __grid_constant__ SelectParams p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    SelectSmem &sm = *reinterpret_cast<SelectSmem *>(smem_raw);
    const int r = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t k = p.k;
    if (tid == 0) {
        sm.n_sure = 0;
        sm.n_cand = 0;
    }

    // the request's own inputs (its store view, start and table length) can
    // be read before the scoring kernel ends: only keys and lengths are its
    const int64_t start = p.place ? (int64_t)p.start_pos[r] : 0;
    const int32_t tl = p.place ? p.table_lens[r] : 0;
    const kvi_store_view st = load_store(p.store, r);
    const bool ok = !p.store.many || store_ok(st, p.g, p.max_facts, k);
    pdl_wait();  // keys and lengths of the scoring kernel
    pdl_launch_dependents();
    const int64_t N = ok ? (p.cand ? (int64_t)p.cand_n[r] : st.n_facts) : 0;
    const uint64_t *keys = p.keys + (int64_t)r * p.key_stride;
    const int32_t *lens = p.lens + (int64_t)r * p.key_stride;
    // up to kSelectThreads * kKeysPerThread keys (and their lengths) are read
    // once, in one round trip, and kept in registers; larger stores stream
    // them from L2
    const bool in_regs = N <= (int64_t)kSelectThreads * kKeysPerThread;
    // larger stores, up to the launcher's allowance: one pass keeps each
    // key's top 16 bits in shared memory, so that the threshold and the
    // candidates need no second read of the keys from L2 (candidates fetch
    // their full key and length)
    const bool in_smem = !in_regs && N <= (int64_t)p.smem_keys;
    uint16_t *hs = reinterpret_cast<uint16_t *>(smem_raw + sizeof(SelectSmem));
    uint64_t kr[kKeysPerThread];
    int32_t lr[kKeysPerThread];
    if (in_regs) {
#pragma unroll
        for (int m = 0; m < kKeysPerThread; ++m) {
            const int64_t i = tid + (int64_t)m * kSelectThreads;
            kr[m] = i < N ? __ldcg(keys + i) : 0;
            lr[m] = i < N ? __ldcg(lens + i) : -1;
        }
    }

    // Fast path.  The top 16 bits of a key, h, are monotone in it.  The keys
    // are split into 256 disjoint groups (4 threads' keys each).  Let t* be
    // the largest t such that at least k groups hold a key with h >= t: then
    // at least k keys have h >= t*, and any key with h < t* has k keys above
    // it, so the top k all have h >= t*.  The groups' largest h go to shared
    // memory and one warp finds t* (kth_largest_bound, no block barriers);
    // the keys with h >= t* are collected (typically little more than k) and
    // ranked exactly.  If more than kCandCap keys qualify (heavy ties),
    // select_by_histogram runs instead.
    bool fast = false;
    if (ok) {
        uint32_t mt = 0;  // this thread's largest h (0 also when it has no key)
        static_assert(kSelectThreads / 4 == kSelectGroups, "groups of 4 threads");
        if (in_regs) {
#pragma unroll
            for (int m = 0; m < kKeysPerThread; ++m) mt = max(mt, (uint32_t)(kr[m] >> 48));
        } else if (in_smem) {
            // kStreamUnroll loads in flight per thread
            for (int64_t i0 = tid; i0 < N; i0 += (int64_t)kStreamUnroll * kSelectThreads) {
                uint64_t v[kStreamUnroll];
#pragma unroll
                for (int u = 0; u < kStreamUnroll; ++u) {
                    const int64_t i = i0 + (int64_t)u * kSelectThreads;
                    v[u] = i < N ? __ldcg(keys + i) : 0;
                }
#pragma unroll
                for (int u = 0; u < kStreamUnroll; ++u) {
                    const int64_t i = i0 + (int64_t)u * kSelectThreads;
                    if (i < N) {
                        const uint32_t h = (uint32_t)(v[u] >> 48);
                        hs[i] = (uint16_t)h;
                        mt = max(mt, h);
                    }
                }
            }
        } else {
            for (int64_t i = tid; i < N; i += kSelectThreads) mt = max(mt, (uint32_t)(__ldcg(keys + i) >> 48));
        }
        // groups of 4 threads (256 groups): group g = threads 4g .. 4g+3
        mt = max(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
        mt = max(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
        if ((lane & 3) == 0) sm.hist[tid >> 2] = mt;
        __syncthreads();
        if (warp == 0) {
            // t = 0 qualifies whenever fewer than k groups hold keys: then
            // every key becomes a candidate
            uint32_t v[kSelectGroups / 32];
#pragma unroll
            for (int i = 0; i < kSelectGroups / 32; ++i) v[i] = sm.hist[i * 32 + lane];
            const uint32_t t_star = kth_largest_bound(v, (uint32_t)k);
            if (lane == 0) sm.bucket = t_star;
        }
        __syncthreads();
        const uint32_t lo = sm.bucket;
        // this thread's qualifying keys go to one warp-aggregated slot range
        // (keys past N are 0 and lo >= 1 unless every key is a candidate)
        uint32_t cnt = 0;
        if (in_regs) {
#pragma unroll
            for (int m = 0; m < kKeysPerThread; ++m)
                cnt += (tid + (int64_t)m * kSelectThreads < N && (uint32_t)(kr[m] >> 48) >= lo) ? 1u : 0u;
        } else if (in_smem) {
            for (int64_t i = tid; i < N; i += kSelectThreads) cnt += (uint32_t)hs[i] >= lo ? 1u : 0u;
        } else {
            for (int64_t i = tid; i < N; i += kSelectThreads)
                cnt += ((uint32_t)(__ldcg(keys + i) >> 48) >= lo) ? 1u : 0u;
        }
        uint32_t incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        uint32_t base = 0;
        if (lane == 31 && incl) base = atomicAdd(&sm.n_cand, incl);
        uint32_t at = __shfl_sync(0xffffffffu, base, 31) + incl - cnt;
        if (cnt) {
            if (in_regs) {
#pragma unroll
                for (int m = 0; m < kKeysPerThread; ++m) {
                    const int64_t i = tid + (int64_t)m * kSelectThreads;
                    if (i < N && (uint32_t)(kr[m] >> 48) >= lo) {
                        if (at < (uint32_t)kCandCap) {
                            sm.cand_key[at] = kr[m];
                            sm.cand_id[at] = (int32_t)i;
                            sm.cand_len[at] = lr[m];
                        }
                        ++at;
                    }
                }
            } else if (in_smem) {
                for (int64_t i = tid; i < N; i += kSelectThreads) {
                    if ((uint32_t)hs[i] >= lo) {
                        if (at < (uint32_t)kCandCap) {
                            sm.cand_key[at] = __ldcg(keys + i);
                            sm.cand_id[at] = (int32_t)i;
                            sm.cand_len[at] = __ldcg(lens + i);
                        }
                        ++at;
                    }
                }
            } else {
                for (int64_t i = tid; i < N; i += kSelectThreads) {
                    const uint64_t key = __ldcg(keys + i);
                    if ((uint32_t)(key >> 48) >= lo) {
                        if (at < (uint32_t)kCandCap) {
                            sm.cand_key[at] = key;
                            sm.cand_id[at] = (int32_t)i;
                            sm.cand_len[at] = __ldcg(lens + i);
                        }
                        ++at;
                    }
                }
            }
        }
        __syncthreads();
        const uint32_t C = sm.n_cand;
        fast = C <= (uint32_t)kCandCap;
        if (fast) {
            for (uint32_t c = warp; c < C; c += kSelectThreads / 32) {
                const uint64_t kc = sm.cand_key[c];
                const int32_t ic = sm.cand_id[c];
                const uint32_t rank = warp_rank(sm.cand_key, sm.cand_id, C, kc, ic, lane);
                if (lane == 0 && rank < (uint32_t)k) {
                    sm.out_key[rank] = kc;
                    sm.out_id[rank] = ic;
                    sm.out_len[rank] = sm.cand_len[c];
                }
            }
        } else {
            // the fallback starts from a zero histogram, empty lists and
            // cleared outputs
            for (int b = tid; b < kHistBins; b += kSelectThreads) sm.hist[b] = 0;
            for (int e = tid; e < KVI_MAX_K; e += kSelectThreads) {
                sm.sure_key[e] = 0;
                sm.sure_id[e] = -1;
                sm.sure_len[e] = -1;
                sm.out_key[e] = 0;
                sm.out_id[e] = -1;
                sm.out_len[e] = -1;
            }
            if (tid == 0) sm.n_cand = 0;
        }
        __syncthreads();
    }
    if (ok && !fast) select_by_histogram(sm, keys, lens, N, k);
    if (ok && p.cand) {
        // shared-store path: ranks were taken over candidate slots, whose
        // order is the fact ids' order; map the slots to fact ids
        for (int j = tid; j < k; j += kSelectThreads)
            sm.out_id[j] = __ldcg(p.cand + (int64_t)r * p.key_stride + sm.out_id[j]);
        __syncthreads();
    }

    for (int j = tid; j < k; j += kSelectThreads) {
        p.ids[(int64_t)r * k + j] = ok ? sm.out_id[j] : -1;
        p.scores[(int64_t)r * k + j] =
            ok ? key_score(sm.out_key[j]) : __int_as_float(0x7fc00000);
        // retrieval-only calls: a selected fact whose extent the scorer
        // found outside the store is reported (placement reports it itself)
        if (!p.place && ok && sm.out_len[j] < 0) record_status(p.status, KVI_ERR_OUT_OF_RANGE);
    }
    if (p.place) {
        place_parallel(p, sm, r, ok, st, start, tl);
        if (r == 0 && tid == 0) *p.work = 0ull;  // the inject kernel's work counter
    }
}

// ------------------------------------------------------ shared-store path

// One CTA per query: t* = the largest t such that at least k of 256 groups
// of facts hold a lo whose key's top 16 bits are >= t (so at least k facts
// have lo >= T = the smallest value with those bits, i.e. T is at most the
// k-th largest lo, itself at most the k-th largest exact score); every fact
// with hi >= T is a candidate, and no other fact can be in the top k.  The
// bound holds for any split of the facts into disjoint groups.  Each warp
// owns a contiguous segment of ids and its lanes read consecutive facts
// (coalesced, kCandUnroll loads in flight per lane); a group is 4 lanes'
// facts.  Candidates are written in id order: a block scan over the warps'
// counts gives each segment its base, and ballots order each warp's facts.
// Twelve loads in flight per lane cover a 10k-fact row of lo or hi in one
// round trip (about 2 us less per 64-query call than four).
constexpr int kCandUnroll = 12;

__global__ void __launch_bounds__(kSelectThreads, 1) cand_kernel(const __grid_constant__ CandParams p)
{
    __shared__ uint32_t gmax[kSelectGroups];
    __shared__ uint32_t wtot[32];
    __shared__ uint32_t t_star;
    constexpr int kWarps = kSelectThreads / 32;
    const int r = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait();  // the intervals of the coarse kernel
    pdl_launch_dependents();
    const float *lo = p.lo + (int64_t)r * p.stride;
    const float *hi = p.hi + (int64_t)r * p.stride;
    const int64_t N = p.N;
    // warp segments of whole 32-fact rows
    const int64_t rows = (N + 31) / 32;
    const int64_t per = (rows + kWarps - 1) / kWarps;
    const int64_t s0 = min(N, (int64_t)warp * per * 32), s1 = min(N, s0 + per * 32);
    uint32_t mt = 0;
    for (int64_t b = s0; b < s1; b += 32 * kCandUnroll) {
        float v[kCandUnroll];
#pragma unroll
        for (int u = 0; u < kCandUnroll; ++u) {
            const int64_t i = b + 32 * u + lane;
            v[u] = i < s1 ? __ldcg(lo + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kCandUnroll; ++u)
            if (b + 32 * u + lane < s1) mt = max(mt, order32(v[u]) >> 16);
    }
    mt = max(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = max(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    if ((lane & 3) == 0) gmax[tid >> 2] = mt;
    __syncthreads();
    if (warp == 0) {
        uint32_t v[kSelectGroups / 32];
#pragma unroll
        for (int i = 0; i < kSelectGroups / 32; ++i) v[i] = gmax[i * 32 + lane];
        const uint32_t a = kth_largest_bound(v, (uint32_t)p.k);  // t = 0 admits every fact
        if (lane == 0) t_star = a;
    }
    __syncthreads();
    const uint32_t T = t_star << 16;
    // this warp's count, then its base among the warps (segments in order)
    uint32_t cnt = 0;
    for (int64_t b = s0; b < s1; b += 32 * kCandUnroll) {
        float v[kCandUnroll];
#pragma unroll
        for (int u = 0; u < kCandUnroll; ++u) {
            const int64_t i = b + 32 * u + lane;
            v[u] = i < s1 ? __ldcg(hi + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kCandUnroll; ++u)
            cnt += __popc(__ballot_sync(0xffffffffu, b + 32 * u + lane < s1 && order32(v[u]) >= T));
    }
    if (lane == 0) wtot[warp] = cnt;
    __syncthreads();
    uint32_t base = 0, total = 0;
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t c = wtot[w];
        base += w < warp ? c : 0u;
        total += c;
    }
    int32_t *cand = p.cand + (int64_t)r * p.stride;
    uint32_t at = base;
    for (int64_t b = s0; b < s1; b += 32 * kCandUnroll) {
        float v[kCandUnroll];
#pragma unroll
        for (int u = 0; u < kCandUnroll; ++u) {
            const int64_t i = b + 32 * u + lane;
            v[u] = i < s1 ? __ldcg(hi + i) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kCandUnroll; ++u) {
            const int64_t i = b + 32 * u + lane;
            const bool take = i < s1 && order32(v[u]) >= T;
            const unsigned m = __ballot_sync(0xffffffffu, take);
            if (take) cand[at + __popc(m & ((1u << lane) - 1u))] = (int32_t)i;
            at += __popc(m);
        }
    }
    if (tid == 0) p.cand_n[r] = (int32_t)total;
}

// Exact keys of the candidates: one warp per candidate, the same Dot2
// accumulation, combination and warp reduction as the scoring kernels, so a
// candidate's key is bit for bit the key the plain path computes for it.
constexpr int kRescoreWarps = 8;
constexpr int kRescoreBlocksPerQuery = 16;

__global__ void __launch_bounds__(kRescoreWarps * 32) rescore_kernel(const __grid_constant__ RescoreParams p)
{
    const int r = blockIdx.y;
    const int lane = threadIdx.x & 31;
    const int E = p.store.g.embed_dim;
    pdl_wait();  // the candidates
    pdl_launch_dependents();
    const int32_t n = p.cand_n[r];
    const float4 *q4 = reinterpret_cast<const float4 *>(p.queries + (int64_t)r * E);
    for (int64_t j = (int64_t)blockIdx.x * kRescoreWarps + (threadIdx.x >> 5); j < n;
         j += (int64_t)gridDim.x * kRescoreWarps) {
        const int32_t f = __ldg(p.cand + (int64_t)r * p.stride + j);
        const float4 *row = reinterpret_cast<const float4 *>(p.store.emb + (int64_t)f * E);
        int64_t s0 = 0;
        int32_t l0 = -1;
        if (lane == 1) {
            s0 = __ldg(p.store.fact_start + f);
            l0 = __ldg(p.store.fact_len + f);
        }
        Dot2x4 acc;
        acc.zero();
#pragma unroll 4
        for (int v = lane; v < E / 4; v += 32) acc.add(__ldg(q4 + v), ld_stream_f4(row + v));
        float s, c;
        acc.combine(s, c);
        warp_reduce_pair(s, c);
        const int64_t at = (int64_t)r * p.stride + j;
        if (lane == 0) p.keys[at] = score_key(s, c);
        if (lane == 1) p.lens[at] = (l0 >= 0 && s0 >= 0 && s0 + l0 <= p.store.n_tokens) ? l0 : -1;
    }
}

// ---------------------------------------------------------------- placement

__global__ void __launch_bounds__(32) place_kernel(const __grid_constant__ PlaceParams p)
{
    const int lane = threadIdx.x;
    const int per = (p.n + 31) / 32;
    const int j0 = lane * per;
    int64_t run = 0;
    for (int m = 0; m < per && j0 + m < p.n; ++m) {
        const int32_t f = p.ids[j0 + m];
        if (f >= 0 && (int64_t)f < p.store.n_facts) run += max(0, p.store.fact_len[f]);
        else record_status(p.status, KVI_ERR_OUT_OF_RANGE);
    }
    int64_t incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    int64_t at = p.start + incl - run;
    for (int m = 0; m < per && j0 + m < p.n; ++m) {
        const int32_t f = p.ids[j0 + m];
        p.pos[j0 + m] = (int32_t)at;
        if (f >= 0 && (int64_t)f < p.store.n_facts) at += max(0, p.store.fact_len[f]);
    }
    if (lane == 31 && p.start + incl > 0x7fffffff) record_status(p.status, KVI_ERR_OUT_OF_RANGE);
}

template <int NV>
cudaError_t launch_score_nv(const ScoreParams &p, cudaStream_t s)
{
    DeviceInfo di;
    cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    const int64_t rows = (int64_t)p.R * p.max_facts;
    const int64_t warps = (rows + 1) / 2;  // at least two rows per warp
    const int64_t cap = (int64_t)di.sms * 2 * (kScoreThreads / 32);
    const int64_t w = warps < cap ? warps : cap;
    const unsigned blocks = (unsigned)((w + kScoreThreads / 32 - 1) / (kScoreThreads / 32));
    score_kernel<NV><<<blocks, kScoreThreads, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score(const ScoreParams &p, cudaStream_t s)
{
    const int E = p.g.embed_dim;
    if (E * 4 <= 8192) {
        DeviceInfo di;
        cudaError_t e = device_info(&di);
        if (e != cudaSuccess) return e;
        const int smem = (int)sizeof(ScoreRingSmem);
        e = smem_opt_in(score_ring_kernel, smem);
        if (e != cudaSuccess) return e;
        const int64_t rows = (int64_t)p.R * p.max_facts;
        const int64_t blocks = rows < di.sms ? rows : di.sms;
        score_ring_kernel<<<(unsigned)blocks, kRingThreads, smem, s>>>(p);
        return cudaGetLastError();
    }
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

cudaError_t prepare_retrieval_kernels()
{
    cudaError_t e = smem_opt_in(score_ring_kernel, (int)sizeof(ScoreRingSmem));
    if (e != cudaSuccess) return e;
    return smem_opt_in(select_kernel, (int)(sizeof(SelectSmem) + 2 * kSmemKeysMax));
}

cudaError_t launch_select(const SelectParams &p0, cudaStream_t s, bool pdl)
{
    SelectParams p = p0;
    // the row space of a request: its keys' stride (facts, or candidate
    // slots of the shared-store path)
    const int64_t rows = p.key_stride;
    p.smem_keys = (rows > (int64_t)kSelectThreads * kKeysPerThread && rows <= kSmemKeysMax) ? (int32_t)rows : 0;
    const int smem = (int)(sizeof(SelectSmem) + (((size_t)p.smem_keys * 2 + 15) & ~(size_t)15));
    cudaError_t e = smem_opt_in(select_kernel, (int)(sizeof(SelectSmem) + 2 * kSmemKeysMax));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.R);
    cfg.blockDim = dim3(kSelectThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    e = cudaLaunchKernelEx(&cfg, select_kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

namespace {

// A launch that may begin while the previous kernel of the stream runs (it
// waits for that kernel's memory itself).
template <typename P>
cudaError_t launch_pdl(void (*kernel)(P), const P &p, dim3 grid, dim3 block, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_candidates(const CandParams &p, cudaStream_t s, bool pdl)
{
    return launch_pdl(cand_kernel, p, dim3((unsigned)p.R), dim3(kSelectThreads), s, pdl);
}

cudaError_t launch_rescore(const RescoreParams &p, cudaStream_t s, bool pdl)
{
    return launch_pdl(rescore_kernel, p, dim3(kRescoreBlocksPerQuery, (unsigned)p.R), dim3(kRescoreWarps * 32), s,
                      pdl);
}

cudaError_t launch_place(const PlaceParams &p, cudaStream_t s)
{
    place_kernel<<<1, 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvi

#ifdef KVI_DEBUG_CHECKS
#include "kvi_debug.h"

extern "C" kvi_status kvi_debug_stall_scorer_row(int64_t row)
{
    const long long v = row < 0 ? -1 : (long long)row;
    const cudaError_t e = cudaMemcpyToSymbol(kvi::g_debug_stall_row, &v, sizeof v);
    if (e != cudaSuccess) return kvi::set_error(KVI_ERR_CUDA, cudaGetErrorString(e));
    return KVI_OK;
}
#endif

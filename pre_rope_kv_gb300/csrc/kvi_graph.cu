// Graph index kernels ("InferScale: GPU-Native KV Injection for Personalized
// LLM Serving", review Summary: retrieval through a GPU ANN index, Jasper;
// Axiom & Free-Parameter Ledger: 64 neighbours, beam width 64; reference
// list: CAGRA's best-first search from a candidate buffer).
//
//   graph_rows_kernel    turns a batch of shared-store top-(degree + 1)
//                        lists into graph rows (the row's own fact dropped).
//   graph_search_kernel  one CTA per query.  The beam lives in shared
//                        memory, sorted by (key descending, id ascending),
//                        with an expanded flag per entry.  Per iteration:
//                        warp 0 picks the first `width` unexpanded entries
//                        (ballots over the sorted beam); all threads load
//                        the parents' neighbour ids and test-and-set them in
//                        the query's visited bitmap (atomicOr, so each fact
//                        is scored at most once, exactly); each warp scores
//                        a new fact with the same Dot2 keys as the scan; the
//                        new facts and the beam are merged by counting
//                        ranks (ids are distinct, so every rank is unique)
//                        into the other half of a double buffer.
// The search is latency-bound (each iteration waits on a graph row, the
// bitmap and the new rows); throughput comes from many queries in flight.
#include <cuda_runtime.h>

#include "kvi_dot2.cuh"
#include "kvi_internal.cuh"

namespace kvi {
namespace {

// 256 threads per query when many queries share the GPU (4 CTAs per SM);
// 512 when there are too few queries to fill it, so that one query scores
// twice as many new facts per memory round trip
constexpr int kSearchThreadsBatch = 256;
constexpr int kSearchThreadsAlone = 512;

struct SearchSmem {
    uint64_t key[2][KVI_MAX_GRAPH_BEAM];
    int32_t id[2][KVI_MAX_GRAPH_BEAM];
    uint8_t expanded[2][KVI_MAX_GRAPH_BEAM];
    uint64_t new_key[KVI_MAX_GRAPH_FRONTIER];
    int32_t new_id[KVI_MAX_GRAPH_FRONTIER];
    int32_t parent[KVI_MAX_GRAPH_FRONTIER];
    int32_t n_new;
    int32_t n_parent;
};

__global__ void __launch_bounds__(256) graph_rows_kernel(const __grid_constant__ GraphRowsParams p)
{
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= p.R) return;
    const int64_t self = p.i0 + r;
    const int32_t *in = p.ids + (int64_t)r * (p.degree + 1);
    int32_t *out = p.graph + self * p.degree;
    int o = 0;
    for (int j = 0; j <= p.degree && o < p.degree; ++j)
        if (in[j] != self) out[o++] = in[j];
}

// Test-and-set `f` in the visited bitmap; the thread that sets the bit adds
// f to the new list (warp-aggregated slot).  `want` false: no candidate.
__device__ __forceinline__ void visit(SearchSmem &sm, uint32_t *vis, int64_t N, int32_t f, bool want,
                                      int32_t *status)
{
    bool fresh = false;
    if (want) {
        if (f < 0 || (int64_t)f >= N) {
            record_status(status, KVI_ERR_OUT_OF_RANGE);
        } else {
            const uint32_t bit = 1u << (f & 31);
            fresh = !(atomicOr(vis + (f >> 5), bit) & bit);
        }
    }
    const unsigned mask = __ballot_sync(0xffffffffu, fresh);
    if (!mask) return;
    const int lane = threadIdx.x & 31;
    int base = 0;
    if (lane == __ffs(mask) - 1) base = atomicAdd(&sm.n_new, __popc(mask));
    base = __shfl_sync(0xffffffffu, base, __ffs(mask) - 1);
    if (fresh) sm.new_id[base + __popc(mask & ((1u << lane) - 1u))] = f;
}

// Dot2 key of every new fact.  A warp scores ROWS rows at a time, and each
// lane loads up to kRowChunk float4 of each of them before any arithmetic,
// so that a 1024-d row costs one round trip to memory.  ROWS = 2 when one
// CTA runs per query and SM (registers to spare), 1 in batches.
constexpr int kRowChunk = 8;

template <int T, int ROWS>
__device__ __forceinline__ void score_new(const GraphSearchParams &p, SearchSmem &sm, const float *q, int n_new)
{
    constexpr int kSearchWarps = T / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float4 *q4 = reinterpret_cast<const float4 *>(q);
    const int E4 = p.E / 4;
    for (int m0 = ROWS * warp; m0 < n_new; m0 += ROWS * kSearchWarps) {
        const float4 *row[ROWS];
#pragma unroll
        for (int x = 0; x < ROWS; ++x) {
            const int m = min(m0 + x, n_new - 1);  // a missing second row re-reads the first
            const int32_t f = sm.new_id[m];
            row[x] = reinterpret_cast<const float4 *>(p.emb + (int64_t)f * p.E);
            // a scored fact may become a parent: bring its graph row into
            // L2 now, so that expanding it later costs an L2 hit
            if (m == m0 + x && lane * 32 < p.degree)
                asm volatile("prefetch.global.L2 [%0];" ::"l"(p.graph + (int64_t)f * p.degree + lane * 32));
        }
        Dot2x4 acc[ROWS];
#pragma unroll
        for (int x = 0; x < ROWS; ++x) acc[x].zero();
        for (int v0 = 0; v0 < E4; v0 += 32 * kRowChunk) {
            float4 r[ROWS][kRowChunk];
#pragma unroll
            for (int u = 0; u < kRowChunk; ++u) {
                const int v = v0 + lane + 32 * u;
#pragma unroll
                for (int x = 0; x < ROWS; ++x)
                    if (v < E4) r[x][u] = ld_stream_f4(row[x] + v);
            }
#pragma unroll
            for (int u = 0; u < kRowChunk; ++u) {
                const int v = v0 + lane + 32 * u;
                if (v < E4) {
                    const float4 qv = __ldg(q4 + v);
#pragma unroll
                    for (int x = 0; x < ROWS; ++x) acc[x].add(qv, r[x][u]);
                }
            }
        }
#pragma unroll
        for (int x = 0; x < ROWS; ++x) {
            float s, c;
            acc[x].combine(s, c);
            warp_reduce_pair(s, c);
            if (lane == 0 && m0 + x < n_new) sm.new_key[m0 + x] = score_key(s, c);
        }
    }
}

// Merge the beam (cur, nc entries, sorted) with the new facts into the
// other buffer, keeping the best `beam`; returns the new count.  An entry's
// place is the number of entries better than it: among the new facts (a
// count, split over a group of G adjacent lanes and summed by shuffles) plus,
// for a new fact, among the beam (a binary search: the beam is sorted), or
// for a beam entry, its own index.  Ids are distinct, so places are unique.
template <int T>
__device__ __forceinline__ int merge(SearchSmem &sm, int cur, int nc, int n_new, int beam)
{
    constexpr int G = T >= 512 ? 4 : 2;  // lanes per entry
    const int nxt = cur ^ 1;
    const int sub = threadIdx.x & (G - 1);
    const int total = n_new + nc;
    for (int e0 = 0; e0 < total; e0 += T / G) {
        const int e = e0 + (int)threadIdx.x / G;  // the same for the G lanes of a group
        const bool live = e < total;
        uint64_t k = 0;
        int32_t id = 0;
        uint8_t ex = 0;
        if (live) {
            if (e < n_new) {
                k = sm.new_key[e];
                id = sm.new_id[e];
            } else {
                k = sm.key[cur][e - n_new];
                id = sm.id[cur][e - n_new];
                ex = sm.expanded[cur][e - n_new];
            }
        }
        int pos = 0;
        if (live)
            for (int j = sub; j < n_new; j += G) pos += better(sm.new_key[j], sm.new_id[j], k, id) ? 1 : 0;
#pragma unroll
        for (int o = 1; o < G; o <<= 1) pos += __shfl_xor_sync(0xffffffffu, pos, o);
        if (live && sub == 0) {
            if (e < n_new) {
                int lo = 0, hi = nc;  // beam entries better than this one: a prefix
                while (lo < hi) {
                    const int mid = (lo + hi) >> 1;
                    if (better(sm.key[cur][mid], sm.id[cur][mid], k, id)) lo = mid + 1;
                    else hi = mid;
                }
                pos += lo;
            } else {
                pos += e - n_new;
            }
            if (pos < beam) {
                sm.key[nxt][pos] = k;
                sm.id[nxt][pos] = id;
                sm.expanded[nxt][pos] = ex;
            }
        }
    }
    return min(beam, nc + n_new);
}

// batches: 64 registers a thread, 4 CTAs of 256 threads per SM; alone: one
// CTA of 512 threads per SM, up to 128 registers
template <int T>
__global__ void __launch_bounds__(T, T >= 512 ? 1 : 4) graph_search_kernel(const __grid_constant__ GraphSearchParams p)
{
    __shared__ SearchSmem sm;
    const int r = blockIdx.x;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const float *q = p.queries + (int64_t)r * p.E;
    uint32_t *vis = p.visited + (int64_t)r * p.vis_words;
    for (int64_t w = tid; w < p.vis_words; w += T) vis[w] = 0u;
    if (tid == 0) sm.n_new = 0;
    __syncthreads();

    // seeds
    for (int t0 = 0; t0 < p.n_seeds; t0 += T) {
        const int t = t0 + tid;
        visit(sm, vis, p.N, t < p.n_seeds ? p.seeds[(int64_t)r * p.n_seeds + t] : 0, t < p.n_seeds,
              p.status);
    }
    __syncthreads();
    int n_new = sm.n_new;
    score_new<T, (T >= 512 ? 2 : 1)>(p, sm, q, n_new);
    __syncthreads();
    int cur = 0;
    int nc = merge<T>(sm, cur ^ 1, 0, n_new, p.beam);  // into buffer 0 from an empty beam
    __syncthreads();

    int iters = 0;
    int scored = n_new;
    while (iters < p.max_iters) {
        if (warp == 0) {
            // the first `width` unexpanded entries of the beam, in order
            int np = 0;
            for (int base = 0; base < nc && np < p.width; base += 32) {
                const int i = base + lane;
                const bool open = i < nc && !sm.expanded[cur][i];
                const unsigned mask = __ballot_sync(0xffffffffu, open);
                const int rank = np + __popc(mask & ((1u << lane) - 1u));
                if (open && rank < p.width) {
                    sm.expanded[cur][i] = 1;
                    sm.parent[rank] = sm.id[cur][i];
                }
                np = min(p.width, np + __popc(mask));
            }
            if (lane == 0) {
                sm.n_parent = np;
                sm.n_new = 0;
            }
        }
        __syncthreads();
        const int np = sm.n_parent;
        if (np == 0) break;
        ++iters;
        const int total = np * p.degree;
        for (int t0 = 0; t0 < total; t0 += T) {
            const int t = t0 + tid;
            int32_t f = 0;
            if (t < total) f = __ldg(p.graph + (int64_t)sm.parent[t / p.degree] * p.degree + t % p.degree);
            visit(sm, vis, p.N, f, t < total, p.status);
        }
        __syncthreads();
        n_new = sm.n_new;
        scored += n_new;
        score_new<T, (T >= 512 ? 2 : 1)>(p, sm, q, n_new);
        __syncthreads();
        nc = merge<T>(sm, cur, nc, n_new, p.beam);
        cur ^= 1;
        __syncthreads();
    }

    const int cnt = min(nc, p.k);
    if (p.cand_ids) {
        // the beam, already in rank order, becomes the selector's candidate
        // list: slot j holds the j-th best fact, its key and its length
        // (-1 when its extent lies outside the store, as the scan reports)
        for (int j = tid; j < nc; j += T) {
            const int32_t f = sm.id[cur][j];
            const int64_t at = (int64_t)r * p.cand_stride + j;
            const int64_t s0 = __ldg(p.fact_start + f);
            const int32_t l0 = __ldg(p.fact_len + f);
            p.cand_ids[at] = f;
            p.cand_keys[at] = sm.key[cur][j];
            p.cand_lens[at] = (l0 >= 0 && s0 >= 0 && s0 + l0 <= p.n_tokens) ? l0 : -1;
        }
        if (tid == 0) p.cand_n[r] = nc;
    } else {
        for (int j = tid; j < p.k; j += T) {
            p.ids[(int64_t)r * p.k + j] = j < cnt ? sm.id[cur][j] : -1;
            p.scores[(int64_t)r * p.k + j] = j < cnt ? key_score(sm.key[cur][j]) : __int_as_float(0x7fc00000);
        }
    }
    if (tid == 0) {
        if (p.count) p.count[r] = cnt;
        if (p.stats) {
            p.stats[2 * (int64_t)r] = iters;
            p.stats[2 * (int64_t)r + 1] = scored;
        }
    }
}

}  // namespace

cudaError_t launch_graph_rows(const GraphRowsParams &p, cudaStream_t s)
{
    graph_rows_kernel<<<(unsigned)((p.R + 255) / 256), 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_graph_search(const GraphSearchParams &p, cudaStream_t s)
{
    DeviceInfo di;
    const cudaError_t e = device_info(&di);
    if (e != cudaSuccess) return e;
    if (p.R <= di.sms) graph_search_kernel<kSearchThreadsAlone><<<(unsigned)p.R, kSearchThreadsAlone, 0, s>>>(p);
    else graph_search_kernel<kSearchThreadsBatch><<<(unsigned)p.R, kSearchThreadsBatch, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace kvi

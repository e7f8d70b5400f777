// kvi_internal.cuh -- declarations shared by the library's translation units
// (host API, retrieval kernels, inject kernel).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kvi.h"

namespace kvi {

// ---------------------------------------------------------------- constants
constexpr int kHistBins = 4096;     // first-level score buckets per request
constexpr int kScoreThreads = 256;  // 8 warps, one fact row per warp at a time
constexpr int kSelectThreads = 1024;
constexpr int kKeysPerThread = 12;  // keys a select thread keeps in registers
constexpr int kCandCap = 1024;      // candidates ranked directly in shared memory
constexpr int kInjConsumers = 12;   // inject warps that rotate / write pieces
constexpr int kInjThreads = (kInjConsumers + 1) * 32;  // + one producer warp
constexpr int kInjRing = 24;        // shared-memory stages per inject CTA
constexpr int kPieceMax = 8192;     // bytes of one staged piece
constexpr int kMaxPrefix = 4096;    // requests (fused) or facts (split) per inject call
constexpr int kMaxRequests = KVI_MAX_REQUESTS;
static_assert(KVI_MAX_REQUESTS <= kMaxPrefix && KVI_MAX_INJECT_FACTS <= kMaxPrefix, "prefix");

// A store is either one host-provided view (single-request calls) or a device
// array of views indexed by request (fused batched call).
struct StoreRef {
    kvi_store_view single;
    const kvi_store_view *many;
};

// Workspace regions (byte offsets from the workspace base, 256-aligned).
// Nothing in it needs initialising: every region is written before it is read
// within one call.
struct WsLayout {
    size_t keys;      // uint64 [R][key_stride] order-preserving score keys
    size_t lens;      // int32  [R][key_stride] validated fact length, -1 = bad extent
    size_t slot_len;  // int32  [R][k] length of each selected fact
    size_t pc;        // int32  [R][k + 1] piece prefix of the selected facts
    size_t npc;       // int32  [R] pieces of each request (0: nothing to inject)
    size_t rows;      // int64  [R][k] first store row of each selected fact
    size_t work;      // uint64 [1] next inject item to hand out (zeroed by select)
    size_t total;
    int64_t key_stride;
};
WsLayout ws_layout(int32_t R, int64_t max_facts, int32_t k);

// How the inject kernel cuts facts into pieces that fit one shared-memory
// stage: `ct` tokens (a divisor of the page size, so a piece never crosses a
// page) of `hg` heads; a token splits into `units` = H / hg head groups when
// one token row is larger than a stage.
struct PieceGeom {
    int32_t ct, hg, units;
};
PieceGeom piece_geom(int32_t H, int32_t D, int32_t block_size);

struct ScoreParams {
    StoreRef store;
    const float *queries;  // [R][E]
    kvi_geometry g;
    int32_t R, k;
    int64_t max_facts;
    uint64_t *keys;
    int32_t *lens;
    int64_t key_stride;
    int32_t *status;  // device status word (first error wins)
};

struct SelectParams {
    StoreRef store;
    kvi_geometry g;
    int32_t R, k;
    int64_t max_facts;
    int64_t key_stride;
    const uint64_t *keys;
    const int32_t *lens;
    // shared-store path: keys[r][j] belong to fact cand[r][j] (ids ascending)
    // for j < cand_n[r]; null for the plain path (keys[r][i] = fact i)
    const int32_t *cand;
    const int32_t *cand_n;
    int32_t *ids;     // [R][k]
    float *scores;    // [R][k]
    // placement (fused path only; place == 0 skips it)
    int32_t place;
    const int32_t *start_pos;   // [R]
    const int32_t *table_lens;  // [R]
    int32_t max_blocks;
    int32_t block_size;
    PieceGeom pg;
    int32_t *pos;               // [R][k]
    int32_t *slot_len;          // [R][k]
    int32_t *pc;                // [R][k + 1]
    int32_t *npc;               // [R]
    int64_t *rows;              // [R][k] first store row of each selected fact
    unsigned long long *work;   // inject work counter, zeroed here
    int32_t *status;
    int32_t smem_keys;          // set by the launcher: keys the CTA may stage in shared memory
};

struct PlaceParams {
    kvi_store_view store;
    const int32_t *ids;
    int32_t n;
    int32_t start;
    int32_t *pos;
    int32_t *status;
};

struct InjectParams {
    StoreRef store;
    int32_t L, H, D;
    PieceGeom pg;
    int32_t fused;             // 0: n explicit facts; 1: R requests of k facts
    const int32_t *ids;        // split [n], fused [R][k]
    const int32_t *pos;        // split [n] start positions, fused [R][k]
    int32_t n;                 // split
    int32_t R, k;              // fused
    const int32_t *slot_len;   // fused [R][k]
    const int32_t *pc;         // fused [R][k + 1]
    const int32_t *npc;        // fused [R]
    const int64_t *rows;       // fused [R][k] first store row of each fact
    unsigned long long *work;  // fused: shared item counter (dynamic balance); split: null
    const int32_t *block_tables;  // split [table_len], fused [R][max_blocks]
    const int32_t *table_lens;    // fused [R]
    int32_t table_len;            // split
    int32_t max_blocks;           // fused row stride
    int32_t num_blocks, block_size;
    const float4 *rope;        // [rope_positions][D/2]: pairs of frequencies, see kvi_host.cu
    int32_t rope_positions;
    int32_t pairing;           // KVI_ROPE_PAIR_*
    int32_t *status;
    void *layer_base[KVI_MAX_LAYERS];
};

// Shared-store scoring (kvi_shared.cu): tensor-core coarse scores with a
// guaranteed interval [lo, hi] around every exact score.
struct CoarseParams {
    int32_t N, R, Rp, E;       // facts, queries, queries padded to 16, embedding dim
    int32_t stages, tmem_cols; // set by the launcher
    int32_t mt;                // accumulators (128-fact tiles) per CTA: 1 or 2
    int32_t box_q;             // query rows per tensor copy (set by the launcher)
    int32_t F;                 // split form: facts per tile (the MMA's N), a multiple of 16, <= 256
    int32_t split;             // split form: CTAs (one cluster) sharing a tile, each a K range
    int64_t stride;            // row stride of lo / hi
    float *lo, *hi;            // [R][stride]
    int32_t *status;
};
cudaError_t launch_coarse(const CoarseParams &p, const float *emb, int64_t n_facts, const float *queries,
                          cudaStream_t s);

// Per query r: candidates = facts whose hi reaches a lower bound of the k-th
// largest lo, in id order (cand[r][0..cand_n[r])); then their exact keys.
struct CandParams {
    const float *lo, *hi;
    int64_t stride;
    int32_t N, R, k;
    int32_t *cand, *cand_n;
};
cudaError_t launch_candidates(const CandParams &p, cudaStream_t s, bool pdl);

struct RescoreParams {
    kvi_store_view store;
    const float *queries;  // [R][E]
    int32_t R;
    int64_t stride;
    const int32_t *cand, *cand_n;
    uint64_t *keys;
    int32_t *lens;
};
cudaError_t launch_rescore(const RescoreParams &p, cudaStream_t s, bool pdl);

// Graph index: the neighbour rows of a build batch (a row's top degree + 1
// ids without the row's own fact) and the beam search, one CTA per query.
struct GraphRowsParams {
    const int32_t *ids;  // [R][degree + 1] top ids of rows i0 .. i0 + R - 1
    int64_t i0;
    int32_t R, degree;
    int32_t *graph;      // [N][degree]
};
cudaError_t launch_graph_rows(const GraphRowsParams &p, cudaStream_t s);

struct GraphSearchParams {
    const float *emb;       // [N][E]
    int64_t N;
    int32_t E;
    const int32_t *graph;   // [N][degree]
    int32_t degree;
    const float *queries;   // [R][E]
    const int32_t *seeds;   // [R][n_seeds]
    int32_t R, n_seeds, beam, width, max_iters, k;
    int32_t *ids;           // [R][k]
    float *scores;          // [R][k]
    int32_t *count;         // [R] or null
    int32_t *stats;         // [R][2] (iterations, facts scored) or null
    uint32_t *visited;      // [R][vis_words] bitmaps
    int64_t vis_words;
    int32_t *status;
    // fused calls: the final beam as the selector's candidates (slots in
    // rank order), with exact keys and validated lengths; ids/scores unused
    int32_t *cand_ids;      // [R][cand_stride] or null
    uint64_t *cand_keys;
    int32_t *cand_lens;
    int32_t *cand_n;        // [R]
    int64_t cand_stride;
    const int64_t *fact_start;
    const int32_t *fact_len;
    int64_t n_tokens;
};
cudaError_t launch_graph_search(const GraphSearchParams &p, cudaStream_t s);

// Diagnostic: a wait on a barrier nothing completes, bounded by limit_ns.
cudaError_t launch_bounded_wait(uint64_t limit_ns, int32_t *status, int64_t *elapsed_ns, cudaStream_t s);
// Diagnostic: the SMs read `bytes` at src (device or mapped host memory).
cudaError_t launch_stream_read(const void *src, size_t bytes, int ctas_per_sm, uint64_t *sum, cudaStream_t s);

// One-time per-device kernel attributes (shared-memory opt-in), made ahead
// of a stream capture.
cudaError_t prepare_retrieval_kernels();
cudaError_t prepare_inject_kernel();

// Launchers (return the CUDA error of the launch).  `pdl` launches the kernel
// with programmatic stream serialization so that it can start while the
// previous kernel of the stream drains; the kernel waits for that kernel's
// results before reading them.
cudaError_t launch_score(const ScoreParams &p, cudaStream_t s);
cudaError_t launch_select(const SelectParams &p, cudaStream_t s, bool pdl);
cudaError_t launch_place(const PlaceParams &p, cudaStream_t s);
cudaError_t launch_inject(const InjectParams &p, cudaStream_t s, bool pdl);
#ifdef KVI_DEBUG_CHECKS
// Debug builds: record KVI_ERR_INVALID_ARG when two facts of a split inject
// call target overlapping positions.
cudaError_t launch_overlap_check(const InjectParams &p, cudaStream_t s);
#endif

// Record a message for kvi_last_error() on this thread and return `s`.
kvi_status set_error(kvi_status s, const char *msg);
// The store checks kvi_retrieve_topk applies (geometry, n_facts, emb).
kvi_status check_retrieval_store(const kvi_store_view *s);
// The checks of a store used for retrieval and injection (emb, kv, extents).
kvi_status check_full_store(const kvi_store_view *s);
// The library's compile-time geometry limits (records a message on failure).
kvi_status check_store_geometry(const kvi_geometry *g);

// Device facts cached per device (SM count).
struct DeviceInfo {
    int sms;
};
cudaError_t device_info(DeviceInfo *out);

// Raise a kernel's dynamic shared-memory limit to `bytes`, once per device
// and kernel (later calls only look the pair up).
cudaError_t smem_opt_in_raw(const void *kernel, int bytes);
template <typename K>
inline cudaError_t smem_opt_in(K kernel, int bytes)
{
    return smem_opt_in_raw(reinterpret_cast<const void *>(kernel), bytes);
}

// Device-side helpers shared by the kernels.
#ifdef __CUDACC__
__device__ __forceinline__ void record_status(int32_t *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}
// Programmatic dependent launch: wait for the previous kernel's memory, and
// let the next kernel of the stream begin launching.  Both are no-ops when
// the kernel was launched without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

}  // namespace kvi

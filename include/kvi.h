/*
 * kvi.h -- C ABI of the GB300 (sm_103a) retrieve-and-inject library.
 *
 * The operation is the serving-time path of "InferScale: GPU-Native KV
 * Injection for Personalized LLM Serving" (pith.science review of arXiv
 * 2607.27090):
 *   - Figure 2 caption: every memory fact is stored twice under one fact_id,
 *     as a retrieval embedding and as pre-RoPE key/value tensors; at serving
 *     time the top-k retrieved facts are resolved to their KV and positioned
 *     by Chunked RoPE;
 *   - Section 5.1 / Theorem 6 (Chunked RoPE): keys are kept before rotary
 *     encoding and rotated to their serving positions on injection, which is
 *     exact because R_a^T R_b = R_{b-a};
 *   - Section 3.4 (KV-connector premise): the engine allocates paged blocks
 *     for the memory prefix without prefilling them and the K/V are
 *     scatter-copied into them before the forward pass.
 *
 * Conventions of this library (readings where the page is silent):
 *   - similarity = dot product of float32 vectors, accumulated so that the
 *     selection key is float64-accurate; exact top-k, ties to the lower id;
 *   - rotary pairing is rotate-half (element i with i + D/2), frequency
 *     omega_i = theta^(-2i/D), angle p * omega_i for token position p;
 *   - retrieved facts are placed back to back, in rank order, from the
 *     request's start position.
 *
 * Memory and ownership.  Every pointer named d_* or described as "device"
 * is device memory owned by the caller and only borrowed for the enqueued
 * work; the library never frees or keeps it.  The only state the library
 * owns is a per-device table of RoPE cos/sin values (see kvi_prepare_rope).
 * All compute calls are asynchronous on the given stream and never
 * synchronise it; results and device-side status are valid once the stream
 * reaches that point.
 *
 * Errors.  A call first validates its host-visible arguments and returns a
 * status without enqueuing anything when they are wrong.  Data-dependent
 * problems that only the GPU can see (a fact id >= n_facts, a block id
 * outside the pool, a position beyond the block table) are recorded in the
 * caller's device word *d_status (the first error wins, via compare-and-swap;
 * the library never clears it) and the offending item is skipped: no kernel
 * writes out of bounds, traps or waits.  kvi_last_error() returns a message
 * for the calling thread's last failing call.
 *
 * Layouts (row-major, innermost last):
 *   store K/V   kv[L][2][n_tokens][H][D]  bf16, index 0 = K (pre-RoPE), 1 = V
 *   embeddings  emb[n_facts][E]           float32
 *   fact extent fact_start[n_facts] int64 (first store row), fact_len int32
 *   paged cache one buffer per layer,     bf16 [2][num_blocks][B][H][D]
 *               (vLLM's flash-attention layout, K then V)
 *   block table block_table[table_len]    int32 block ids, position p lives in
 *               block block_table[p / B] at offset p % B.
 */
#ifndef KVI_H
#define KVI_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KVI_API __attribute__((visibility("default")))
#else
#define KVI_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA handles, ABI-compatible with cudaStream_t / cudaEvent_t. */
typedef struct CUstream_st *kvi_stream_t;
typedef struct CUevent_st *kvi_event_t;

typedef enum {
    KVI_OK = 0,
    KVI_ERR_INVALID_ARG = 1,  /* bad pointer, size, geometry or limit */
    KVI_ERR_OUT_OF_RANGE = 2, /* fact id, store row, block id or position out of range */
    KVI_ERR_CAPACITY = 3,     /* the facts do not fit the request's block table */
    KVI_ERR_CUDA = 4,         /* a CUDA runtime call failed (see kvi_last_error) */
    KVI_ERR_TIMEOUT = 5,      /* a kernel's bounded wait for its own copies expired */
    KVI_ERR_IO = 6            /* a store file could not be written or read, or is not a valid one */
} kvi_status;

/* Compile-time limits of the library. */
#define KVI_MAX_LAYERS 128        /* L */
#define KVI_MAX_K 256             /* facts retrieved per request */
#define KVI_MAX_INJECT_FACTS 4096 /* facts per kvi_inject_paged call */
#define KVI_MAX_REQUESTS 4096     /* requests per kvi_retrieve_and_inject call */
#define KVI_MAX_HEAD_DIM 512      /* D, a multiple of 16 */
#define KVI_MAX_EMBED_DIM 8192    /* E, a multiple of 4 */
#define KVI_MAX_SHARED_QUERIES 256 /* queries per shared-store call */

typedef struct {
    int32_t layers;    /* L */
    int32_t kv_heads;  /* H, KV heads (GQA) */
    int32_t head_dim;  /* D, multiple of 16, <= KVI_MAX_HEAD_DIM */
    int32_t embed_dim; /* E, multiple of 4, <= KVI_MAX_EMBED_DIM */
} kvi_geometry;

/* A fact store (Figure 2 caption: retrieval embedding and pre-RoPE K/V under
 * one fact_id; fact_id = index).  The struct itself lives in host memory for
 * the single-request calls and in device memory (an array of R of them) for
 * kvi_retrieve_and_inject; the pointers inside are device pointers.
 *
 * flags & KVI_STORE_KV_HOST: kv lives in host memory that the GPU reads in
 * place -- pinned host memory (cudaHostAlloc, cudaHostRegister) through
 * its unified address, or any memory on a system with hardware address
 * translation.  The paper keeps a store that outgrows HBM in host DRAM
 * ("a few ms" of extra TTFT); on a Grace host the inject kernel then reads
 * each piece of K/V over NVLink-C2C directly into the rotating warps
 * instead of staging it in shared memory.  emb, fact_start and fact_len stay
 * in device memory. */
#define KVI_STORE_KV_HOST 1u
typedef struct {
    kvi_geometry g;
    int64_t n_facts;           /* N */
    int64_t n_tokens;          /* rows per (layer, K|V) plane of kv */
    const void *kv;            /* bf16 [L][2][n_tokens][H][D] */
    const float *emb;          /* float32 [N][E] */
    const int64_t *fact_start; /* [N] first store row of each fact */
    const int32_t *fact_len;   /* [N] tokens of each fact, >= 0; both extents
                                * are required by every call, since the
                                * scoring kernels validate each fact's */
    uint32_t flags;            /* KVI_STORE_* */
    uint32_t reserved;         /* 0 */
} kvi_store_view;

typedef struct {
    int64_t n_tokens;      /* total rows = sum of fact_len */
    size_t kv_bytes;       /* L * 2 * n_tokens * H * D * 2 */
    size_t emb_bytes;      /* N * E * 4 */
    size_t offsets_bytes;  /* (N + 1) * 8 */
} kvi_store_sizes;

/* The engine's paged KV pool (Section 3.4): one device buffer per layer,
 * each bf16 [2][num_blocks][block_size][H][D].  layer_base is a HOST array
 * of `layers` device pointers, read during the call only. */
typedef struct {
    void *const *layer_base;
    int32_t layers;
    int32_t num_blocks;
    int32_t block_size; /* B, tokens per block */
} kvi_paged_cache;

/* Store layout (host only, no device work).  Dense CSR layout of a store
 * whose facts are written back to back: token_offsets_out[i] = sum of
 * fact_len[0..i), token_offsets_out[n_facts] = n_tokens, plus the byte sizes
 * of the buffers the caller allocates.  fact_len (host, [n_facts]) must be
 * >= 0.  token_offsets_out (host, [n_facts + 1]) may be NULL.  Errors:
 * KVI_ERR_INVALID_ARG for a bad geometry, n_facts < 0 or a negative length. */
KVI_API kvi_status kvi_store_layout(const kvi_geometry *g, const int32_t *fact_len,
                            int64_t n_facts, int64_t *token_offsets_out,
                            kvi_store_sizes *sizes_out);

/* Build (or extend) this device's RoPE table for (rope_theta, head_dim)
 * covering positions [0, max_position).  cos/sin of p * omega_i are
 * computed in float64 on the host and kept as hi/lo float32 pairs, so that
 * the kernels rotate bf16 keys to within one rounding of the exact result at
 * any position (Section 5.1, Chunked RoPE).  Synchronous; allocates device
 * memory owned by the library until process exit.  The inject calls build
 * the table on first use when needed, which blocks the host and is refused
 * (KVI_ERR_INVALID_ARG) while the stream is being captured; call this first
 * to keep them asynchronous.
 * Lifetime: no table is freed before the process exits.  When a call needs
 * more positions than the current table covers, a table with at least twice
 * the rows replaces it for later calls; the old one stays allocated, so
 * kernels already enqueued and plans recorded earlier (which hold its
 * address) keep reading valid memory.  Neither this call nor the growth
 * synchronises the device.
 * Errors: KVI_ERR_INVALID_ARG (theta <= 0, head_dim not a multiple of 16,
 * max_position <= 0 or > 2^22), KVI_ERR_CUDA. */
KVI_API kvi_status kvi_prepare_rope(double rope_theta, int32_t head_dim,
                            int32_t max_position);

/* Rotary-encoding variants.  The paper names only "rotary position
 * embedding" (RoFormer); the plain calls above and below use rotate-half
 * pairing with omega_i = theta^(-2i/D).  A kvi_rope selects the other
 * conventions a serving engine may use, so that injected keys match the
 * engine's own query rotation:
 *   pairing  KVI_ROPE_PAIR_HALF        element i pairs with i + D/2
 *                                      (Llama, Mistral, Qwen);
 *            KVI_ROPE_PAIR_INTERLEAVED element 2i pairs with 2i + 1
 *                                      (GPT-J, RoFormer's original form);
 *   scaling  KVI_ROPE_SCALE_NONE       omega_i = theta^(-2i/D);
 *            KVI_ROPE_SCALE_LLAMA3     Llama 3.1 scaling of those
 *                                      frequencies: with wavelength
 *                                      w = 2 pi / omega, components with
 *                                      w < original / high_freq_factor keep
 *                                      omega, those with w > original /
 *                                      low_freq_factor use omega / factor,
 *                                      and in between the two are blended
 *                                      linearly in original / w;
 *   table    cos_table/sin_table (host float32 [table_positions][D/2], pair
 *            i at column i) with table_id != 0: the engine's own
 *            coefficients, used as given (theta and scaling are ignored).
 *            The library copies a table the first time it sees table_id on
 *            a device and reuses that copy afterwards: never reuse an id
 *            for other contents.  Positions at or beyond table_positions
 *            are out of range (KVI_ERR_OUT_OF_RANGE on the device).
 * Computed tables keep the float64 hi/lo precision described under
 * kvi_prepare_rope; a caller's table is applied in float32 as given. */
#define KVI_ROPE_PAIR_HALF 0
#define KVI_ROPE_PAIR_INTERLEAVED 1
#define KVI_ROPE_SCALE_NONE 0
#define KVI_ROPE_SCALE_LLAMA3 1
typedef struct {
    double theta;                  /* base, > 0 (unless a table is given) */
    int32_t pairing;               /* KVI_ROPE_PAIR_* */
    int32_t scaling;               /* KVI_ROPE_SCALE_* */
    double factor;                 /* LLAMA3: > 0 (Llama 3.1: 8) */
    double low_freq_factor;        /* LLAMA3: > 0 (1) */
    double high_freq_factor;       /* LLAMA3: > low_freq_factor (4) */
    double original_max_positions; /* LLAMA3: > 0 (8192) */
    const float *cos_table;        /* optional host table, see above */
    const float *sin_table;
    int32_t table_positions;
    int64_t table_id;
} kvi_rope;

/* kvi_prepare_rope for any kvi_rope (head_dim as there).  Errors:
 * KVI_ERR_INVALID_ARG (a field outside the ranges above, a table with
 * table_id == 0 or fewer than max_position rows), KVI_ERR_CUDA. */
KVI_API kvi_status kvi_prepare_rope_ex(const kvi_rope *rope, int32_t head_dim,
                                       int32_t max_position);

/* Device scratch bytes needed by kvi_retrieve_topk (R = 1) and
 * kvi_retrieve_and_inject for R requests of at most max_facts facts and k
 * retrieved facts each.  Returns 0 for invalid sizes. */
KVI_API size_t kvi_workspace_bytes(int32_t R, int64_t max_facts, int32_t k);

/* Retrieve (Figure 2 caption, "top-k retrieved facts"): score every fact
 * embedding against d_query ([E] float32, device) and return the exact
 * top-k under (score descending, fact id ascending).
 *   d_ids    [k] int32, rank order      d_scores [k] float32 similarity
 *   d_ws     scratch of >= kvi_workspace_bytes(1, store->n_facts, k) bytes,
 *            256-byte aligned; its contents need no initialisation.
 *   d_status device int32, required: device-side errors of this call are
 *            recorded there (first error wins; never cleared by the
 *            library): KVI_ERR_OUT_OF_RANGE when a selected fact's extent
 *            (fact_start, fact_len) lies outside the store -- its id is
 *            still returned -- and KVI_ERR_TIMEOUT when a scoring wait gave
 *            up (the ids are then not valid).
 * Errors: KVI_ERR_INVALID_ARG (null pointers, k < 1, k > KVI_MAX_K,
 * k > n_facts, bad geometry, workspace too small), KVI_ERR_CUDA. */
KVI_API kvi_status kvi_retrieve_topk(const kvi_store_view *store, const float *d_query,
                             int32_t k, int32_t *d_ids, float *d_scores,
                             void *d_ws, size_t ws_bytes, int32_t *d_status,
                             kvi_stream_t stream);

/* Place (Figure 2 caption, "positioned by chunked RoPE"; rank-order reading):
 * d_pos[j] = start + sum of fact_len[d_ids[j']] for j' < j.  n <= KVI_MAX_K.
 * An id outside [0, n_facts) records KVI_ERR_OUT_OF_RANGE in *d_status and
 * counts as length 0.  Errors: KVI_ERR_INVALID_ARG, KVI_ERR_CUDA. */
KVI_API kvi_status kvi_place(const kvi_store_view *store, const int32_t *d_ids,
                     int32_t n, int32_t start, int32_t *d_pos,
                     int32_t *d_status, kvi_stream_t stream);

/* Inject (Section 5.1 Chunked RoPE + Section 3.4 scatter-copy): for each of
 * the n facts d_fact_ids[j] ([n] int32, device) and each of its tokens t,
 * rotate the pre-RoPE K rows of every layer and head to position
 * p = d_start_pos[j] + t and write K and V (unchanged) into the paged cache
 * slot (d_block_table[p / B], p % B).  d_block_table: [table_len] int32
 * device.  Positions must not overlap (overlaps are caller error; the
 * result is then unspecified).  n <= KVI_MAX_INJECT_FACTS.  Device-side
 * errors (recorded in *d_status, item skipped): fact id or store row out of
 * range, p < 0 or p >= table_len * B, block id outside [0, num_blocks).
 * Errors: KVI_ERR_INVALID_ARG (null pointers, geometry, cache mismatch,
 * theta <= 0, limits), KVI_ERR_CUDA. */
KVI_API kvi_status kvi_inject_paged(const kvi_store_view *store,
                            const int32_t *d_fact_ids,
                            const int32_t *d_start_pos, int32_t n,
                            const int32_t *d_block_table, int32_t table_len,
                            const kvi_paged_cache *cache, double rope_theta,
                            int32_t *d_status, kvi_stream_t stream);

/* kvi_inject_paged with the rotation given by *rope instead of rope_theta
 * (Section 5.1 Chunked RoPE under another rotary convention; the variants
 * are described at kvi_rope).  Same arguments and errors otherwise. */
KVI_API kvi_status kvi_inject_paged_ex(const kvi_store_view *store,
                                       const int32_t *d_fact_ids,
                                       const int32_t *d_start_pos, int32_t n,
                                       const int32_t *d_block_table, int32_t table_len,
                                       const kvi_paged_cache *cache, const kvi_rope *rope,
                                       int32_t *d_status, kvi_stream_t stream);

/* Fused retrieve + place + inject for R independent requests (Figure 2
 * serving path; Section 6.4's concurrent users).  Request r scores its own
 * store d_stores[r] (device array of R kvi_store_view, all with geometry g)
 * against d_queries[r] ([R][E] float32), keeps the top-k, places them back
 * to back from d_start_pos[r] and injects them through block table row r
 * (d_block_tables [R][max_blocks] int32, d_table_lens [R] int32 <=
 * max_blocks).  Outputs: d_ids, d_scores, d_pos, each [R][k] (rank order).
 *   max_facts  host upper bound of every store's n_facts (sizes the grid);
 *   d_ws       >= kvi_workspace_bytes(R, max_facts, k) bytes, 256-aligned,
 *              no initialisation needed.
 * Device-side errors, recorded in *d_status: a store with n_facts < k or
 * > max_facts, another geometry, or a bad fact extent (KVI_ERR_OUT_OF_RANGE;
 * that request retrieves nothing); facts that do not fit the request's
 * block table (KVI_ERR_CAPACITY; that request injects nothing); block ids
 * outside the pool (KVI_ERR_OUT_OF_RANGE; that token is skipped).
 * Errors: KVI_ERR_INVALID_ARG, KVI_ERR_CUDA. */
KVI_API kvi_status kvi_retrieve_and_inject(
    const kvi_geometry *g, int32_t R, const kvi_store_view *d_stores,
    int64_t max_facts, const float *d_queries, int32_t k,
    const int32_t *d_start_pos, const int32_t *d_block_tables,
    const int32_t *d_table_lens, int32_t max_blocks,
    const kvi_paged_cache *cache, double rope_theta, int32_t *d_ids,
    float *d_scores, int32_t *d_pos, void *d_ws, size_t ws_bytes,
    int32_t *d_status, kvi_stream_t stream);

/* kvi_retrieve_and_inject with the rotation given by *rope instead of
 * rope_theta (variants at kvi_rope).  Same arguments and errors otherwise. */
KVI_API kvi_status kvi_retrieve_and_inject_ex(
    const kvi_geometry *g, int32_t R, const kvi_store_view *d_stores,
    int64_t max_facts, const float *d_queries, int32_t k,
    const int32_t *d_start_pos, const int32_t *d_block_tables,
    const int32_t *d_table_lens, int32_t max_blocks,
    const kvi_paged_cache *cache, const kvi_rope *rope, int32_t *d_ids,
    float *d_scores, int32_t *d_pos, void *d_ws, size_t ws_bytes,
    int32_t *d_status, kvi_stream_t stream);

/* Plans: one fused call recorded once into a CUDA graph and replayed.  A
 * serving loop calls kvi_retrieve_and_inject_ex with the same buffers for
 * every request and only their contents change (query, start, block table).
 * A plan records that call once -- its three kernel launches, with their
 * programmatic dependencies as graph edges -- so that each request costs
 * one graph launch on the host instead of three kernel launches and the
 * argument checks.  The arguments are those of kvi_retrieve_and_inject_ex;
 * the buffers must stay valid, and their contents are read at each
 * kvi_plan_launch.  *d_status is not reset by a launch (as with direct
 * calls, the first error stays).  Creating a plan builds the RoPE table
 * first, records on a private stream and needs no other stream to be idle.
 * Errors: those of kvi_retrieve_and_inject_ex, KVI_ERR_CUDA. */
typedef struct kvi_plan_s *kvi_plan;
KVI_API kvi_status kvi_plan_create_fused(
    kvi_plan *plan, const kvi_geometry *g, int32_t R, const kvi_store_view *d_stores,
    int64_t max_facts, const float *d_queries, int32_t k, const int32_t *d_start_pos,
    const int32_t *d_block_tables, const int32_t *d_table_lens, int32_t max_blocks,
    const kvi_paged_cache *cache, const kvi_rope *rope, int32_t *d_ids, float *d_scores,
    int32_t *d_pos, void *d_ws, size_t ws_bytes, int32_t *d_status);
/* kvi_plan_create_fused that also records the request's copies: before the
 * fused call, in_bytes from pinned host memory h_in to device d_in (the
 * request's packed inputs, e.g. query | start | block table, which the
 * d_* arguments point into); after it, out_bytes from device d_out to
 * pinned host memory h_out (the packed outputs).  A serving loop then
 * writes a request into h_in, launches the plan once and reads h_out after
 * the stream is synchronised.  h_in / h_out must be pinned (cudaHostAlloc or
 * cudaHostRegister); 0 bytes skips that copy. */
KVI_API kvi_status kvi_plan_create_fused_io(
    kvi_plan *plan, const kvi_geometry *g, int32_t R, const kvi_store_view *d_stores,
    int64_t max_facts, const float *d_queries, int32_t k, const int32_t *d_start_pos,
    const int32_t *d_block_tables, const int32_t *d_table_lens, int32_t max_blocks,
    const kvi_paged_cache *cache, const kvi_rope *rope, int32_t *d_ids, float *d_scores,
    int32_t *d_pos, void *d_ws, size_t ws_bytes, int32_t *d_status, const void *h_in,
    void *d_in, size_t in_bytes, const void *d_out, void *h_out, size_t out_bytes);
/* Replay the plan on `stream` (stream order applies as for a kernel). */
KVI_API kvi_status kvi_plan_launch(kvi_plan plan, kvi_stream_t stream);
/* Free the plan (after its last launch has completed). */
KVI_API kvi_status kvi_plan_destroy(kvi_plan plan);

/* Shared-store retrieval: R queries against ONE store (Section 6.4, where
 * concurrent users query one conversation's memory).  Scoring R queries
 * against the same embeddings is the dense contraction S = Q E^T, which runs
 * on the tensor cores (TF32, float32 accumulation) and gives each score an
 * interval that provably contains the exact value.  The facts whose interval
 * can reach the k-th score are then rescored exactly (the same compensated
 * dot product as kvi_retrieve_topk), so the result is the exact top-k under
 * (score descending, fact id ascending): identical to kvi_retrieve_topk run
 * once per query, at one read of the embeddings instead of R.
 *   store      one kvi_store_view (host struct; device pointers inside)
 *   d_queries  [R][E] float32 device, 16-byte aligned;
 *              1 <= R <= KVI_MAX_SHARED_QUERIES
 *   d_ids, d_scores  [R][k] (rank order)
 *   d_ws       >= kvi_workspace_bytes_shared(R, n_facts, k) bytes,
 *              256-byte aligned, no initialisation needed
 *   d_status   device int32 or NULL (a timed-out wait records
 *              KVI_ERR_TIMEOUT)
 * Errors: KVI_ERR_INVALID_ARG, KVI_ERR_CUDA. */
KVI_API size_t kvi_workspace_bytes_shared(int32_t R, int64_t n_facts, int32_t k);
KVI_API kvi_status kvi_retrieve_topk_shared(const kvi_store_view *store, int32_t R,
                                            const float *d_queries, int32_t k, int32_t *d_ids,
                                            float *d_scores, void *d_ws, size_t ws_bytes,
                                            int32_t *d_status, kvi_stream_t stream);

/* kvi_retrieve_and_inject for R requests that share one store: the shared
 * retrieval above, then placement and injection of each request through its
 * own block table row (arguments as in kvi_retrieve_and_inject_ex, with the
 * store as one host kvi_store_view). */
KVI_API kvi_status kvi_retrieve_and_inject_shared(
    const kvi_store_view *store, int32_t R, const float *d_queries, int32_t k,
    const int32_t *d_start_pos, const int32_t *d_block_tables, const int32_t *d_table_lens,
    int32_t max_blocks, const kvi_paged_cache *cache, const kvi_rope *rope, int32_t *d_ids,
    float *d_scores, int32_t *d_pos, void *d_ws, size_t ws_bytes, int32_t *d_status,
    kvi_stream_t stream);

/* No-allocation retrieval.  The paper has no counterpart: this call exists
 * for callers that cannot allocate device memory where they retrieve -- a
 * serving engine that has reserved nearly all GPU memory for its own KV pool
 * and gives a plugin only the buffers of a request, a latency-bound loop that
 * must not call cudaMalloc/cudaFree (they can synchronise the device), or a
 * C caller without an allocator.  It computes exactly what kvi_retrieve_topk
 * computes (same kernels, same results) but keeps its scratch in a fixed
 * array of KVI_NOALLOC_SCRATCH_BYTES of device memory that belongs to the
 * library instead of a caller workspace; it calls no cudaMalloc, cudaFree or
 * allocating library routine.
 *   - The array exists on every GPU that loads the library, until the
 *     process exits.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make
 *     that first call before any stream capture.  The cached address
 *     belongs to the device's context as it was then: after
 *     cudaDeviceReset (or anything else that destroys that context) this
 *     entry point must not be called again in the process.
 *   - All calls on a device share the one array and it keeps whatever the
 *     last call left; nothing in it has to start at zero.  Calls whose work
 *     overlaps on the GPU (other streams, other host threads, or before the
 *     previous call's kernels have finished on an unordered stream) race on
 *     it; order them on one stream.
 *   - n_facts must be <= KVI_NOALLOC_MAX_FACTS; larger stores are rejected
 *     with KVI_ERR_INVALID_ARG (use kvi_retrieve_topk with a workspace).
 * Arguments, outputs and other errors are those of kvi_retrieve_topk. */
#define KVI_NOALLOC_MAX_FACTS 65536
#define KVI_NOALLOC_SCRATCH_BYTES (KVI_NOALLOC_MAX_FACTS * 12 + 65536)
KVI_API kvi_status kvi_retrieve_topk_noalloc(const kvi_store_view *store,
                                             const float *d_query, int32_t k,
                                             int32_t *d_ids, float *d_scores,
                                             int32_t *d_status, kvi_stream_t stream);

/* Graph index.  The review's Summary retrieves facts at serving time
 * through a GPU ANN index (Jasper) rather than a scan, and its Axiom &
 * Free-Parameter Ledger sets the index at 64 graph neighbours and beam width
 * 64; the reference list cites CAGRA, a GPU graph index searched best-first
 * from a buffer of candidates.  Readings of this library (the pages give
 * nothing more):
 *   - the graph links each fact to its `degree` most similar other facts,
 *     exactly (the same score and order as kvi_retrieve_topk: score
 *     descending, ties to the lower id), as int32 graph[N][degree];
 *   - the search keeps a beam of the best `beam` facts scored so far, each
 *     marked expanded or not.  It scores the query's seed facts, then, up to
 *     max_iters times, expands the best `width` unexpanded facts of the beam
 *     (none left: it stops), scores every neighbour of theirs that it has not
 *     scored before and keeps the best `beam` of the beam and the new facts.
 *     No fact is scored twice (an exact visited set).  The result is the
 *     first k facts of the beam, in rank order;
 *   - the seeds are the caller's (e.g. drawn at random), so that a search is
 *     a deterministic function of its inputs.
 * The search is approximate retrieval: its recall against the exact top-k
 * depends on the data, the graph and the parameters. */
#define KVI_MAX_GRAPH_DEGREE 128  /* degree */
#define KVI_MAX_GRAPH_BEAM 256    /* beam */
#define KVI_MAX_GRAPH_FRONTIER 512 /* n_seeds, and width * degree */

/* Device workspace of kvi_graph_build for a store of n_facts facts (0 for
 * arguments outside the limits). */
KVI_API size_t kvi_graph_build_workspace_bytes(int64_t n_facts, int32_t degree);

/* Build the graph of *store (its embeddings; kv is not read) into d_graph,
 * int32 [n_facts][degree], with 1 <= degree <= min(KVI_MAX_GRAPH_DEGREE,
 * n_facts - 1).  Each row's neighbours come from the exact shared-store
 * retrieval (kvi_retrieve_topk_shared) of its own embedding, degree + 1
 * facts, without the row's own fact; batches of KVI_MAX_SHARED_QUERIES rows
 * are enqueued on `stream` one after another.  d_ws: device,
 * kvi_graph_build_workspace_bytes, 256-byte aligned.  Errors:
 * KVI_ERR_INVALID_ARG, KVI_ERR_CUDA; device-side errors in *d_status. */
KVI_API kvi_status kvi_graph_build(const kvi_store_view *store, int32_t degree, int32_t *d_graph,
                                   void *d_ws, size_t ws_bytes, int32_t *d_status,
                                   kvi_stream_t stream);

typedef struct {
    int32_t beam;      /* k <= beam <= KVI_MAX_GRAPH_BEAM */
    int32_t width;     /* >= 1, width * degree <= KVI_MAX_GRAPH_FRONTIER */
    int32_t max_iters; /* >= 0 */
    int32_t n_seeds;   /* 1 .. KVI_MAX_GRAPH_FRONTIER seeds per query */
} kvi_graph_search_params;

/* Device workspace of kvi_graph_search: one visited bitmap of n_facts bits
 * per query (0 for arguments outside the limits). */
KVI_API size_t kvi_graph_search_workspace_bytes(int32_t R, int64_t n_facts);

/* Search the graph d_graph [n_facts][degree] (as kvi_graph_build writes it,
 * or any graph of valid ids) for R queries d_queries [R][E] from the seeds
 * d_seeds [R][n_seeds] (fact ids).  Outputs, device: d_ids [R][k] and
 * d_scores [R][k] in rank order (-1 and NaN past a query's result count);
 * d_count [R] (may be NULL), the number of results, k unless the beam held
 * fewer facts; d_stats [R][2] (may be NULL), the iterations run and the
 * facts scored.  One CTA per query; 1 <= R <= 65535.  d_ws: device,
 * kvi_graph_search_workspace_bytes, 256-byte aligned.  Errors (host):
 * KVI_ERR_INVALID_ARG for bad pointers or parameters; a seed or graph id
 * outside [0, n_facts) is recorded as KVI_ERR_OUT_OF_RANGE in *d_status and
 * skipped. */
KVI_API kvi_status kvi_graph_search(const kvi_store_view *store, const int32_t *d_graph,
                                    int32_t degree, int32_t R, const float *d_queries,
                                    const int32_t *d_seeds, const kvi_graph_search_params *params,
                                    int32_t k, int32_t *d_ids, float *d_scores, int32_t *d_count,
                                    int32_t *d_stats, void *d_ws, size_t ws_bytes,
                                    int32_t *d_status, kvi_stream_t stream);

/* Graph retrieval and injection, fused, for R requests over one store
 * (the pages' serving path with the ANN index: retrieve, rotate by Chunked
 * RoPE, scatter into the paged cache).  Each query is searched as by
 * kvi_graph_search; its final beam, in rank order, is handed to the same
 * selection, placement and inject kernels as kvi_retrieve_and_inject_shared,
 * so the first k facts of the beam are injected back to back from
 * d_start_pos[r] through block table r.  Arguments are those of
 * kvi_graph_search (no counts or stats) and of
 * kvi_retrieve_and_inject_shared; 1 <= R <= KVI_MAX_REQUESTS.  If a beam
 * holds fewer than k facts, the missing ranks come back as id -1 and
 * KVI_ERR_OUT_OF_RANGE is recorded.  d_ws: device,
 * kvi_graph_retrieve_and_inject_workspace_bytes, 256-byte aligned.  Errors:
 * as the two calls named. */
KVI_API size_t kvi_graph_retrieve_and_inject_workspace_bytes(int32_t R, int64_t n_facts, int32_t beam,
                                                             int32_t k);
KVI_API kvi_status kvi_graph_retrieve_and_inject(
    const kvi_store_view *store, const int32_t *d_graph, int32_t degree, int32_t R,
    const float *d_queries, const int32_t *d_seeds, const kvi_graph_search_params *params, int32_t k,
    const int32_t *d_start_pos, const int32_t *d_block_tables, const int32_t *d_table_lens,
    int32_t max_blocks, const kvi_paged_cache *cache, const kvi_rope *rope, int32_t *d_ids,
    float *d_scores, int32_t *d_pos, void *d_ws, size_t ws_bytes, int32_t *d_status,
    kvi_stream_t stream);

/* Store files.  The paper encodes a user's memory facts offline into a
 * long-lived store of pre-RoPE K/V and embeddings, which may sit in host
 * DRAM when it outgrows HBM (the review's Summary: facts are encoded
 * offline, and CPU offload of the KV store costs a few ms of TTFT).  These
 * calls persist a store and load it back into HBM or pinned host memory.
 *
 * File format, version 1 (all integers little-endian; every section starts
 * at a multiple of 4096 bytes and the gaps are zero):
 *   [0, 8)     magic "KVISTORE"
 *   [8, 12)    uint32 version = 1
 *   [12, 16)   uint32 header bytes = 128
 *   [16, 32)   int32 layers, kv_heads, head_dim, embed_dim
 *   [32, 40)   int64 n_facts N
 *   [40, 48)   int64 n_tokens T (rows per (layer, K|V) plane)
 *   [48, 88)   uint64 file offsets of the sections fact_start, fact_len,
 *              emb, kv, and the file size
 *   [88, 96)   uint64 extents hash: FNV-1a 64 over the bytes of the
 *              fact_start section followed by those of the fact_len section
 *   [96, 104)  uint64 payload hash (below) over the emb section followed by
 *              the kv section
 *   [104, 112) uint64 header hash: FNV-1a 64 over bytes [0, 104)
 *   [112, 128) zero
 * Sections: fact_start int64 [N]; fact_len int32 [N]; emb float32 [N][E];
 * kv bf16 [L][2][T][H][D], exactly as in kvi_store_view.
 * FNV-1a 64: h = 0xcbf29ce484222325; per byte b: h = (h ^ b) * 0x100000001b3
 * (mod 2^64).  Payload hash: the payload read as little-endian uint64 words
 * w_0, w_1, ... goes to four lanes (lane j takes the words with index = j
 * mod 4); lane j starts at 0xcbf29ce484222325 + j and takes each word as
 * h_j = (h_j ^ w) * 0x100000001b3; the hash is
 * h_0 ^ rotl(h_1, 16) ^ rotl(h_2, 32) ^ rotl(h_3, 48). */
typedef struct {
    kvi_geometry g;
    int64_t n_facts;  /* N */
    int64_t n_tokens; /* T */
    size_t kv_bytes;  /* L * 2 * T * H * D * 2 */
    size_t emb_bytes; /* N * E * 4 */
} kvi_store_file_info;

/* Write *store to a new file at path (replaced if it exists).  The store is
 * written as it is: all n_tokens rows of kv, including rows no fact
 * references.  kv may be device memory or, with KVI_STORE_KV_HOST, host
 * memory; emb, fact_start and fact_len are device memory.  Synchronous: the
 * data is read with blocking copies, so the work that writes the store must
 * have finished (synchronise its stream first).  Errors:
 * KVI_ERR_INVALID_ARG (a bad view or geometry), KVI_ERR_IO (the file cannot
 * be created or written; a partial file is removed), KVI_ERR_CUDA. */
KVI_API kvi_status kvi_store_save(const char *path, const kvi_store_view *store);

/* Read and check the header of a store file (host only, no CUDA call), so
 * that the caller can size the buffers for kvi_store_load.  Errors:
 * KVI_ERR_INVALID_ARG (NULL argument), KVI_ERR_IO (the file cannot be read,
 * is not a version-1 store file, its header hash does not match, or its
 * size does not match the header). */
KVI_API kvi_status kvi_store_file_info_read(const char *path, kvi_store_file_info *info);

/* Load the store file at path into caller-owned buffers sized by
 * kvi_store_file_info_read: kv (kv_bytes; device memory, or pinned host
 * memory when flags & KVI_STORE_KV_HOST), emb (device, emb_bytes),
 * fact_start (device, N int64) and fact_len (device, N int32).  The fact
 * extents are checked (start >= 0, length >= 0, start + length <= T) and
 * both hashes are verified.  Synchronous.  Errors: KVI_ERR_INVALID_ARG
 * (NULL or misaligned buffer, unknown flag), KVI_ERR_IO (unreadable file,
 * bad header, hash mismatch or bad extent; the buffers then hold
 * unspecified data), KVI_ERR_CUDA. */
KVI_API kvi_status kvi_store_load(const char *path, void *kv, float *emb, int64_t *fact_start,
                                  int32_t *fact_len, uint32_t flags);

/* Diagnostic: one warp waits on a shared-memory barrier that nothing
 * completes, with the bounded wait every staging kernel of this library
 * uses; after limit_ns (1 us .. 1 s) of %globaltimer it gives up, records
 * KVI_ERR_TIMEOUT in *d_status and returns.  *d_elapsed_ns (device, may be
 * NULL) receives the time the wait took.  Shows that a wait which never
 * completes ends with a status the host reads, not a hang.  Asynchronous.
 * Errors: KVI_ERR_INVALID_ARG, KVI_ERR_CUDA. */
KVI_API kvi_status kvi_selftest_bounded_wait(uint64_t limit_ns, int32_t *d_status,
                                             int64_t *d_elapsed_ns, kvi_stream_t stream);

/* Diagnostic: read `bytes` bytes at `src` with the SMs -- 16-byte loads from
 * every thread of a grid of ctas_per_sm CTAs per SM, grid-stride, 8 loads in
 * flight per thread -- and write one 64-bit checksum (the wrapping sum of
 * the words read) to *d_sum.  `src` may be device memory or pinned host
 * memory the device can address (cudaHostAlloc / cudaHostRegister): timed
 * with events, it gives the rate at which the SMs read that memory, the
 * ceiling of the inject kernel's host-resident pieces (KVI_STORE_KV_HOST),
 * which are staged with the same 16-byte loads.  Asynchronous.  Errors:
 * KVI_ERR_INVALID_ARG (NULL pointers, src not 16-byte aligned, bytes not a
 * multiple of 16, ctas_per_sm outside [1, 8]), KVI_ERR_CUDA. */
KVI_API kvi_status kvi_selftest_stream_read(const void *src, size_t bytes, int32_t ctas_per_sm,
                                            uint64_t *d_sum, kvi_stream_t stream);

/* Tracing: when n_events == 3, the calling thread's next
 * kvi_retrieve_and_inject calls record events[0] before the first kernel,
 * events[1] once retrieval and placement are enqueued and events[2] after
 * the inject kernel, on the call's stream, so that the stages can be timed
 * with cudaEventElapsedTime.  n_events == 0 turns tracing off.  The events
 * are created and owned by the caller.  Errors: KVI_ERR_INVALID_ARG. */
KVI_API kvi_status kvi_trace_stages(const kvi_event_t *events, int32_t n_events);

/* Static description of a status code. */
KVI_API const char *kvi_status_str(kvi_status s);

/* Message of the calling thread's last failing call ("" if none). */
KVI_API const char *kvi_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* KVI_H */

// kvi_noalloc.cu -- kvi_retrieve_topk_noalloc: exact top-k retrieval for
// callers that cannot allocate device memory.
//
// Some callers have no way to get scratch memory at the point where they
// retrieve: a serving engine that has reserved (nearly) all of the GPU's
// memory for its own KV pool at start-up and hands plugins only the buffers
// of a request; code running where the CUDA allocator must not be called
// (cudaMalloc and cudaFree may synchronise the device, which a latency-bound
// serving loop cannot afford); or a C caller with no allocator of its own.
// For them, this entry point keeps the scratch that kvi_retrieve_topk would
// take from the caller's workspace in a fixed array in device memory that
// belongs to the library.  It launches the same kernels as
// kvi_retrieve_topk and allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (KVI_NOALLOC_SCRATCH_BYTES) until the process exits.  On
// the host its name is only a stand-in for the device copy, so its device
// address is looked up with cudaGetSymbolAddress, once per device, on that
// device's first call (the address then stays valid for the life of the
// device's context; a cudaDeviceReset ends it).
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>
#include <vector>

#include "kvi_internal.cuh"

namespace {

using namespace kvi;

// Scratch of one retrieval over at most KVI_NOALLOC_MAX_FACTS facts: the
// 64-bit selection keys and validated lengths the scoring kernel writes and
// the selection kernel reads (the same regions as the workspace of
// kvi_retrieve_topk; the placement regions are unused here).
constexpr size_t kKeysBytes = (size_t)KVI_NOALLOC_MAX_FACTS * 8;
constexpr size_t kLensBytes = (size_t)KVI_NOALLOC_MAX_FACTS * 4;
constexpr size_t kTailBytes = 64 * 1024;  // slot lengths, piece prefixes, counters (<= k entries)
static_assert(KVI_NOALLOC_SCRATCH_BYTES == kKeysBytes + kLensBytes + kTailBytes, "scratch size");

static __device__ __align__(256) unsigned char g_topk_scratch[KVI_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
std::vector<void *> g_addr;  // device address of g_topk_scratch per device ordinal

kvi_status cuda_fail(const char *what, cudaError_t e)
{
    char buf[256];
    snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
    return set_error(KVI_ERR_CUDA, buf);
}

kvi_status scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    std::lock_guard<std::mutex> lock(g_mu);
    if ((int)g_addr.size() <= dev) g_addr.resize(dev + 1, nullptr);
    if (!g_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_topk_scratch);  // with `dev` current
        if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress(scratch)", e);
        if (!p) return set_error(KVI_ERR_CUDA, "cudaGetSymbolAddress(scratch) returned NULL");
        g_addr[dev] = p;
    }
    *out = g_addr[dev];
    return KVI_OK;
}

kvi_status bad(const char *msg) { return set_error(KVI_ERR_INVALID_ARG, msg); }

}  // namespace

extern "C" {

kvi_status kvi_retrieve_topk_noalloc(const kvi_store_view *store, const float *d_query, int32_t k,
                                     int32_t *d_ids, float *d_scores, int32_t *d_status,
                                     kvi_stream_t stream)
{
    kvi_status st = check_retrieval_store(store);
    if (st != KVI_OK) return st;
    if (store->n_facts > KVI_NOALLOC_MAX_FACTS)
        return bad("store has more facts than the fixed scratch holds (KVI_NOALLOC_MAX_FACTS); "
                   "use kvi_retrieve_topk with a workspace");
    if (!d_query || (reinterpret_cast<uintptr_t>(d_query) & 15))
        return bad("query must be a 16-byte aligned device pointer");
    if (k < 1 || k > KVI_MAX_K || (int64_t)k > store->n_facts) return bad("k outside [1, min(KVI_MAX_K, n_facts)]");
    if (!d_ids || !d_scores) return bad("ids or scores is NULL");
    if (!d_status || (reinterpret_cast<uintptr_t>(d_status) & 3))
        return bad("status must be a 4-byte aligned device pointer");

    const WsLayout w = ws_layout(1, store->n_facts, k);
    if (w.total > sizeof(g_topk_scratch)) return bad("scratch layout exceeds the fixed array");
    void *base = nullptr;
    st = scratch_address(&base);
    if (st != KVI_OK) return st;
    char *ws = static_cast<char *>(base);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // nothing in the scratch has to start at zero: the scoring kernel writes
    // every key and length that the selection kernel then reads
    ScoreParams sp{};
    sp.store.single = *store;
    sp.store.many = nullptr;
    sp.queries = d_query;
    sp.g = store->g;
    sp.R = 1;
    sp.k = k;
    sp.max_facts = store->n_facts;
    sp.keys = reinterpret_cast<uint64_t *>(ws + w.keys);
    sp.lens = reinterpret_cast<int32_t *>(ws + w.lens);
    sp.key_stride = w.key_stride;
    sp.status = d_status;
    cudaError_t e = launch_score(sp, s);
    if (e != cudaSuccess) return cuda_fail("launch_score", e);
    SelectParams lp{};
    lp.store = sp.store;
    lp.g = store->g;
    lp.R = 1;
    lp.k = k;
    lp.max_facts = store->n_facts;
    lp.key_stride = w.key_stride;
    lp.keys = sp.keys;
    lp.lens = sp.lens;
    lp.ids = d_ids;
    lp.scores = d_scores;
    lp.place = 0;
    lp.status = d_status;
    e = launch_select(lp, s, true);
    if (e != cudaSuccess) return cuda_fail("launch_select", e);
    return KVI_OK;
}

}  // extern "C"

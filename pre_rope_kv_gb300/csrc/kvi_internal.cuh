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
constexpr int kScoreRowsPerWarp = 4;
constexpr int kSelectThreads = 1024;
constexpr int kCandCap = 1024;      // candidates ranked directly in shared memory
constexpr int kInjectThreads = 256;
constexpr int kLayerGroup = 8;      // layers handled by one inject work item
constexpr int kMaxRequests = 1 << 16;

// A store is either one host-provided view (single-request calls) or a device
// array of views indexed by request (fused batched call).
struct StoreRef {
    kvi_store_view single;
    const kvi_store_view *many;
};

// Workspace regions (byte offsets from the workspace base, 256-aligned).
struct WsLayout {
    size_t hist;     // uint32 [R][kHistBins]
    size_t counter;  // uint32 [1] CTAs of the select kernel that finished
    size_t keys;     // uint64 [R][key_stride] order-preserving score keys
    size_t cum;      // int32  [R][k + 1] token prefix of the selected facts
    size_t tok;      // int64  [R] tokens injected per request
    size_t req_off;  // int64  [R + 1] token offset of each request
    size_t total;
    int64_t key_stride;
};
WsLayout ws_layout(int32_t R, int64_t max_facts, int32_t k);
// Bytes at the start of the workspace that must be zero before each call.
inline size_t ws_zero_bytes(const WsLayout &w) { return w.keys; }

struct ScoreParams {
    StoreRef store;
    const float *queries;  // [R][E]
    kvi_geometry g;
    int32_t R;
    int64_t max_facts;
    int32_t rows_per_cta;
    uint64_t *keys;
    int64_t key_stride;
    uint32_t *hist;
};

struct SelectParams {
    StoreRef store;
    kvi_geometry g;
    int32_t R, k;
    int64_t max_facts;
    int64_t key_stride;
    const uint64_t *keys;
    const uint32_t *hist;
    int32_t *ids;     // [R][k]
    float *scores;    // [R][k]
    // placement (fused path only; place == 0 skips it)
    int32_t place;
    const int32_t *start_pos;   // [R]
    const int32_t *table_lens;  // [R]
    int32_t max_blocks;
    int32_t block_size;
    int32_t *pos;               // [R][k]
    int32_t *cum;               // [R][k + 1]
    int64_t *tok;               // [R]
    int64_t *req_off;           // [R + 1]
    uint32_t *counter;
    int32_t *status;
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
    int32_t fused;             // 0: n explicit facts; 1: R requests of k facts
    const int32_t *ids;        // split [n], fused [R][k]
    const int32_t *pos;        // split [n] start positions, fused [R][k]
    int32_t n;                 // split
    int32_t R, k;              // fused
    const int32_t *cum;        // fused [R][k + 1]
    const int64_t *req_off;    // fused [R + 1]
    const int32_t *block_tables;  // split [table_len], fused [R][max_blocks]
    const int32_t *table_lens;    // fused [R]
    int32_t table_len;            // split
    int32_t max_blocks;           // fused row stride
    int32_t num_blocks, block_size;
    const float4 *rope;        // [rope_positions][D/2] {cos_hi, cos_lo, sin_hi, sin_lo}
    int32_t rope_positions;
    int32_t *status;
    void *layer_base[KVI_MAX_LAYERS];
};

// Launchers (return the CUDA error of the launch).
cudaError_t launch_score(const ScoreParams &p, cudaStream_t s);
cudaError_t launch_select(const SelectParams &p, cudaStream_t s);
cudaError_t launch_place(const PlaceParams &p, cudaStream_t s);
cudaError_t launch_inject(const InjectParams &p, cudaStream_t s);

// Device facts cached per device (SM count, resident inject CTAs per SM).
struct DeviceInfo {
    int sms;
    int inject_ctas_per_sm;
};
cudaError_t device_info(DeviceInfo *out);

}  // namespace kvi

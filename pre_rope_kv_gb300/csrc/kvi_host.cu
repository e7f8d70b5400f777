// kvi_host.cu -- the C ABI: argument validation, workspace layout, the
// per-device RoPE table, and the launch sequences of the four calls.
//
// Path ("InferScale: GPU-Native KV Injection for Personalized LLM Serving"):
// retrieve the top-k facts for a query (Figure 2 caption), position them by
// Chunked RoPE (Section 5.1 / Theorem 6) and scatter-copy their K/V into the
// engine's paged blocks (Section 3.4).  Every step runs in this library's
// kernels; the host only validates, sizes grids and enqueues.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "kvi_internal.cuh"

using namespace kvi;

namespace {

constexpr int32_t kMaxRopePositions = 1 << 22;

thread_local std::string t_last_error;
thread_local cudaEvent_t t_trace[3] = {nullptr, nullptr, nullptr};
thread_local int t_trace_n = 0;

kvi_status fail(kvi_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

#define KVI_CUDA(call)                                                              \
    do {                                                                            \
        const cudaError_t e_ = (call);                                              \
        if (e_ != cudaSuccess)                                                      \
            return fail(KVI_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_));     \
    } while (0)

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kvi_status check_geometry(const kvi_geometry *g)
{
    if (!g) return fail(KVI_ERR_INVALID_ARG, "geometry is NULL");
    if (g->layers < 1 || g->layers > KVI_MAX_LAYERS)
        return fail(KVI_ERR_INVALID_ARG, "layers=%d outside [1, %d]", g->layers, KVI_MAX_LAYERS);
    if (g->kv_heads < 1 || g->kv_heads > 4096)
        return fail(KVI_ERR_INVALID_ARG, "kv_heads=%d outside [1, 4096]", g->kv_heads);
    if (g->head_dim < 16 || g->head_dim > KVI_MAX_HEAD_DIM || g->head_dim % 16)
        return fail(KVI_ERR_INVALID_ARG, "head_dim=%d must be a multiple of 16 in [16, %d]",
                    g->head_dim, KVI_MAX_HEAD_DIM);
    if (g->embed_dim < 4 || g->embed_dim > KVI_MAX_EMBED_DIM || g->embed_dim % 4)
        return fail(KVI_ERR_INVALID_ARG, "embed_dim=%d must be a multiple of 4 in [4, %d]",
                    g->embed_dim, KVI_MAX_EMBED_DIM);
    return KVI_OK;
}

kvi_status check_store(const kvi_store_view *s, bool retrieval, bool inject)
{
    if (!s) return fail(KVI_ERR_INVALID_ARG, "store is NULL");
    kvi_status st = check_geometry(&s->g);
    if (st != KVI_OK) return st;
    if (s->n_facts < 1 || s->n_facts > 0x7fffffff)
        return fail(KVI_ERR_INVALID_ARG, "n_facts=%lld outside [1, 2^31)", (long long)s->n_facts);
    if (s->n_tokens < 0) return fail(KVI_ERR_INVALID_ARG, "n_tokens < 0");
    if (retrieval && (!s->emb || !aligned(s->emb, 16)))
        return fail(KVI_ERR_INVALID_ARG, "emb must be a 16-byte aligned device pointer");
    // every kernel that scores a fact also validates its extent, so the
    // extents are required even by retrieval-only calls
    if (!s->fact_len || !s->fact_start)
        return fail(KVI_ERR_INVALID_ARG, "fact_start and fact_len are required");
    if (inject && (!s->kv || !aligned(s->kv, 16)))
        return fail(KVI_ERR_INVALID_ARG, "kv (16-byte aligned) is required");
    return KVI_OK;
}

kvi_status check_cache(const kvi_paged_cache *c, const kvi_geometry &g)
{
    if (!c || !c->layer_base) return fail(KVI_ERR_INVALID_ARG, "cache or cache->layer_base is NULL");
    if (c->layers != g.layers)
        return fail(KVI_ERR_INVALID_ARG, "cache has %d layers, store %d", c->layers, g.layers);
    if (c->num_blocks < 1 || c->block_size < 1)
        return fail(KVI_ERR_INVALID_ARG, "num_blocks and block_size must be >= 1");
    for (int l = 0; l < c->layers; ++l)
        if (!c->layer_base[l] || !aligned(c->layer_base[l], 16))
            return fail(KVI_ERR_INVALID_ARG, "layer_base[%d] is NULL or not 16-byte aligned", l);
    return KVI_OK;
}

// ------------------------------------------------------------- device facts

std::mutex g_dev_mu;
std::vector<DeviceInfo> g_dev;  // indexed by device ordinal; sms == 0 = unknown

// ---------------------------------------------------------------- RoPE table

// One device table per (device, head_dim, frequencies): the pairing does not
// change the table, only how the kernel applies it.
//
// Lifetime: a table is never freed while the library is loaded.  When a
// call needs more positions than the current table holds, a larger table
// (at least twice the rows) replaces it for later calls and the old one
// moves to g_rope_retired.  Kernels already enqueued, and CUDA graphs
// recorded by kvi_plan_create_fused*, keep the old pointer in their
// parameters; the old table stays valid and covers the positions they were
// recorded for, so no replay reads freed memory and no call has to
// synchronise the device to retire a table.  Doubling bounds the retired
// tables' total size by the current table's.
struct RopeEntry {
    int device;
    int32_t head_dim;
    kvi_rope key;  // theta, scaling and its parameters, or table_id
    int32_t positions;
    float4 *table;
};
std::mutex g_rope_mu;
std::vector<RopeEntry> g_rope;
std::vector<float4 *> g_rope_retired;  // superseded tables, kept until exit

// The last table this thread was handed, looked up without the mutex (the
// pointer stays valid: tables are never freed).
struct RopeHit {
    bool valid;
    int device;
    int32_t head_dim;
    kvi_rope key;
    int32_t positions;
    const float4 *table;
};
thread_local RopeHit t_rope_hit = {false, 0, 0, {}, 0, nullptr};

bool same_table(const kvi_rope &a, const kvi_rope &b)
{
    if (a.table_id || b.table_id) return a.table_id == b.table_id;
    if (a.theta != b.theta || a.scaling != b.scaling) return false;
    return a.scaling == KVI_ROPE_SCALE_NONE ||
           (a.factor == b.factor && a.low_freq_factor == b.low_freq_factor &&
            a.high_freq_factor == b.high_freq_factor &&
            a.original_max_positions == b.original_max_positions);
}

kvi_rope plain_rope(double theta)
{
    kvi_rope r{};
    r.theta = theta;
    r.pairing = KVI_ROPE_PAIR_HALF;
    r.scaling = KVI_ROPE_SCALE_NONE;
    return r;
}

bool finite_pos(double x) { return x > 0.0 && std::isfinite(x); }

kvi_status check_rope(const kvi_rope *r)
{
    if (!r) return fail(KVI_ERR_INVALID_ARG, "rope is NULL");
    if (r->pairing != KVI_ROPE_PAIR_HALF && r->pairing != KVI_ROPE_PAIR_INTERLEAVED)
        return fail(KVI_ERR_INVALID_ARG, "rope pairing=%d is not a KVI_ROPE_PAIR_* value", r->pairing);
    if (r->cos_table || r->sin_table || r->table_id) {
        if (!r->cos_table || !r->sin_table || r->table_id == 0 || r->table_positions <= 0 ||
            r->table_positions > kMaxRopePositions)
            return fail(KVI_ERR_INVALID_ARG,
                        "a rope table needs cos_table, sin_table, table_id != 0 and "
                        "table_positions in [1, 2^22]");
        return KVI_OK;
    }
    if (!finite_pos(r->theta)) return fail(KVI_ERR_INVALID_ARG, "rope theta must be finite and > 0");
    if (r->scaling == KVI_ROPE_SCALE_LLAMA3) {
        if (!finite_pos(r->factor) || !finite_pos(r->low_freq_factor) ||
            !finite_pos(r->high_freq_factor) || !finite_pos(r->original_max_positions) ||
            !(r->high_freq_factor > r->low_freq_factor))
            return fail(KVI_ERR_INVALID_ARG,
                        "LLAMA3 rope scaling needs factor, low_freq_factor, "
                        "original_max_positions > 0 and high_freq_factor > low_freq_factor");
    } else if (r->scaling != KVI_ROPE_SCALE_NONE) {
        return fail(KVI_ERR_INVALID_ARG, "rope scaling=%d is not a KVI_ROPE_SCALE_* value", r->scaling);
    }
    return KVI_OK;
}

// Frequencies omega_i, i < D/2: theta^(-2i/D), optionally with the Llama 3.1
// scaling (components by wavelength: kept, divided by `factor`, or blended
// linearly in original / wavelength between the two edges).
std::vector<double> rope_omega(const kvi_rope &r, int32_t D)
{
    const int32_t half = D / 2;
    std::vector<double> omega(half);
    const double two_pi = 2.0 * std::acos(-1.0);
    for (int32_t i = 0; i < half; ++i) {
        const double w = std::pow(r.theta, -2.0 * (double)i / (double)D);
        double out = w;
        if (r.scaling == KVI_ROPE_SCALE_LLAMA3) {
            const double wavelength = two_pi / w;
            const double short_edge = r.original_max_positions / r.high_freq_factor;
            const double long_edge = r.original_max_positions / r.low_freq_factor;
            if (wavelength > long_edge) {
                out = w / r.factor;
            } else if (wavelength >= short_edge) {
                const double g = (r.original_max_positions / wavelength - r.low_freq_factor) /
                                 (r.high_freq_factor - r.low_freq_factor);
                out = g * w + (1.0 - g) * (w / r.factor);
            }
        }
        omega[i] = out;
    }
    return omega;
}

// Round a double to 16 significant bits (head) and keep the float32 tail.
void split16(double x, float &hi, float &lo)
{
    float f = (float)x;
    uint32_t u;
    std::memcpy(&u, &f, 4);
    u = (u + 0x80u) & 0xffffff00u;
    std::memcpy(&hi, &u, 4);
    lo = (float)(x - (double)hi);
}

// Rows [p0, p1) of the device table: two adjacent frequencies per 32 bytes,
// the layout the kernels read as packed float32 pairs:
// {cos_hi[i], cos_hi[i+1], cos_lo[i], cos_lo[i+1]},
// {sin_hi[i], sin_hi[i+1], sin_lo[i], sin_lo[i+1]}, i even.  A caller's
// table is taken as given: hi = its value, lo = 0.
void fill_rope_rows(const double *omega, const kvi_rope *tab, int32_t D, int32_t p0, int32_t p1,
                    float4 *out)
{
    const int32_t half = D / 2;
    for (int32_t p = p0; p < p1; ++p) {
        for (int32_t i = 0; i < half; i += 2) {
            float ch[2], cl[2], sh[2], sl[2];
            for (int u = 0; u < 2; ++u) {
                if (tab) {
                    ch[u] = tab->cos_table[(size_t)p * half + i + u];
                    sh[u] = tab->sin_table[(size_t)p * half + i + u];
                    cl[u] = sl[u] = 0.0f;
                } else {
                    const double a = (double)p * omega[i + u];
                    split16(std::cos(a), ch[u], cl[u]);
                    split16(std::sin(a), sh[u], sl[u]);
                }
            }
            out[(size_t)p * half + i] = make_float4(ch[0], ch[1], cl[0], cl[1]);
            out[(size_t)p * half + i + 1] = make_float4(sh[0], sh[1], sl[0], sl[1]);
        }
    }
}

// Returns the table of the current device covering >= needed positions (a
// caller's table covers its own rows, whatever is needed).
kvi_status rope_get(const kvi_rope &spec, int32_t D, int32_t needed, cudaStream_t stream,
                    const float4 **table, int32_t *positions)
{
    int dev = 0;
    KVI_CUDA(cudaGetDevice(&dev));
    const bool given = spec.table_id != 0;
    if (given) needed = spec.table_positions;
    RopeHit &th = t_rope_hit;
    if (th.valid && th.device == dev && th.head_dim == D && th.positions >= needed &&
        same_table(th.key, spec)) {
        *table = th.table;
        *positions = th.positions;
        return KVI_OK;
    }
    std::lock_guard<std::mutex> lock(g_rope_mu);
    RopeEntry *hit = nullptr;
    for (auto &e : g_rope)
        if (e.device == dev && e.head_dim == D && same_table(e.key, spec)) hit = &e;
    if (hit && hit->positions >= needed) {
        *table = hit->table;
        *positions = hit->positions;
        th = RopeHit{true, dev, D, hit->key, hit->positions, hit->table};
        return KVI_OK;
    }
    if (stream) {
        cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
        KVI_CUDA(cudaStreamIsCapturing(stream, &cap));
        if (cap != cudaStreamCaptureStatusNone)
            return fail(KVI_ERR_INVALID_ARG,
                        "RoPE table for theta=%g, D=%d, %d positions is missing during stream "
                        "capture; call kvi_prepare_rope first", spec.theta, D, needed);
    }
    int32_t P = given ? needed : std::min(kMaxRopePositions, ((needed + 1023) / 1024) * 1024);
    if (hit && !given)  // grow geometrically: few retired tables, bounded in size
        P = std::max(P, (int32_t)std::min<int64_t>(kMaxRopePositions, 2 * (int64_t)hit->positions));
    const int32_t half = D / 2;
    const std::vector<double> omega = given ? std::vector<double>() : rope_omega(spec, D);
    std::vector<float4> host((size_t)P * half);
    const unsigned hw = std::max(1u, std::min(16u, std::thread::hardware_concurrency()));
    const int32_t nthr = (int32_t)std::min<unsigned>(hw, (unsigned)((P + 1023) / 1024));
    std::vector<std::thread> pool;
    for (int32_t t = 0; t < nthr; ++t) {
        const int32_t a = (int32_t)((int64_t)P * t / nthr), b = (int32_t)((int64_t)P * (t + 1) / nthr);
        pool.emplace_back(fill_rope_rows, omega.data(), given ? &spec : nullptr, D, a, b, host.data());
    }
    for (auto &th : pool) th.join();
    float4 *d = nullptr;
    KVI_CUDA(cudaMalloc(&d, host.size() * sizeof(float4)));
    const cudaError_t ce = cudaMemcpy(d, host.data(), host.size() * sizeof(float4), cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) {
        cudaFree(d);
        return fail(KVI_ERR_CUDA, "RoPE table upload: %s", cudaGetErrorString(ce));
    }
    if (hit) {
        // enqueued kernels and recorded plans may still read the old table:
        // it is retired, not freed (see RopeEntry)
        g_rope_retired.push_back(hit->table);
        hit->table = d;
        hit->positions = P;
    } else {
        kvi_rope key = spec;
        key.cos_table = key.sin_table = nullptr;  // the copy is kept, not the caller's arrays
        g_rope.push_back(RopeEntry{dev, D, key, P, d});
        hit = &g_rope.back();
    }
    *table = d;
    *positions = P;
    th = RopeHit{true, dev, D, hit->key, P, d};
    return KVI_OK;
}

int32_t clamp_rope(int64_t needed)
{
    return (int32_t)std::max<int64_t>(1, std::min<int64_t>(needed, kMaxRopePositions));
}

}  // namespace

// --------------------------------------------------------------- internals

namespace kvi {

cudaError_t device_info(DeviceInfo *out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1, DeviceInfo{0});
    if (g_dev[dev].sms == 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        g_dev[dev] = DeviceInfo{sms};
    }
    *out = g_dev[dev];
    return cudaSuccess;
}

kvi_status set_error(kvi_status s, const char *msg) { return fail(s, "%s", msg); }

kvi_status check_retrieval_store(const kvi_store_view *s) { return check_store(s, true, false); }
kvi_status check_full_store(const kvi_store_view *s) { return check_store(s, true, true); }
kvi_status check_store_geometry(const kvi_geometry *g) { return check_geometry(g); }

cudaError_t smem_opt_in_raw(const void *kernel, int bytes)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::mutex mu;
    static std::vector<std::pair<int, const void *>> done;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto &d : done)
        if (d.first == dev && d.second == kernel) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.emplace_back(dev, kernel);
    return e;
}

PieceGeom piece_geom(int32_t H, int32_t D, int32_t block_size)
{
    const int64_t token_bytes = (int64_t)H * D * 2;
    PieceGeom g{1, H, 1};
    if (token_bytes <= kPieceMax) {
        const int64_t most = std::min<int64_t>(block_size, kPieceMax / token_bytes);
        for (int32_t c = 1; c <= most; ++c)
            if (block_size % c == 0) g.ct = c;
    } else {
        g.hg = 1;
        for (int32_t h = 1; h <= H; ++h)
            if (H % h == 0 && (int64_t)h * D * 2 <= kPieceMax) g.hg = h;
        g.units = H / g.hg;
    }
    return g;
}

WsLayout ws_layout(int32_t R, int64_t max_facts, int32_t k)
{
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    WsLayout w{};
    w.key_stride = (max_facts + 31) & ~(int64_t)31;
    size_t at = 0;
    w.keys = at;     at = up(at + (size_t)R * (size_t)w.key_stride * 8);
    w.lens = at;     at = up(at + (size_t)R * (size_t)w.key_stride * 4);
    w.slot_len = at; at = up(at + (size_t)R * (size_t)k * 4);
    w.pc = at;       at = up(at + (size_t)R * (size_t)(k + 1) * 4);
    w.npc = at;      at = up(at + (size_t)R * 4);
    w.rows = at;     at = up(at + (size_t)R * (size_t)k * 8);
    w.work = at;     at = up(at + 8);
    w.total = at;
    return w;
}

// Shared-store calls: the plain regions plus the coarse intervals and the
// candidate lists.
struct SharedWs {
    WsLayout w;
    size_t lo, hi, cand, cand_n, total;
};

SharedWs shared_layout(int32_t R, int64_t n_facts, int32_t k)
{
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    SharedWs x{};
    x.w = ws_layout(R, n_facts, k);
    const size_t plane = (size_t)R * (size_t)x.w.key_stride * 4;
    size_t at = x.w.total;
    x.lo = at;     at = up(at + plane);
    x.hi = at;     at = up(at + plane);
    x.cand = at;   at = up(at + plane);
    x.cand_n = at; at = up(at + (size_t)R * 4);
    x.total = at;
    return x;
}

}  // namespace kvi

// ------------------------------------------------------------------ the ABI

extern "C" {

const char *kvi_status_str(kvi_status s)
{
    switch (s) {
    case KVI_OK: return "ok";
    case KVI_ERR_INVALID_ARG: return "invalid argument";
    case KVI_ERR_OUT_OF_RANGE: return "index out of range";
    case KVI_ERR_CAPACITY: return "facts do not fit the block table";
    case KVI_ERR_CUDA: return "CUDA error";
    case KVI_ERR_TIMEOUT: return "a kernel wait timed out";
    case KVI_ERR_IO: return "store file error";
    }
    return "unknown status";
}

const char *kvi_last_error(void) { return t_last_error.c_str(); }

kvi_status kvi_store_layout(const kvi_geometry *g, const int32_t *fact_len, int64_t n_facts,
                            int64_t *token_offsets_out, kvi_store_sizes *sizes_out)
{
    kvi_status st = check_geometry(g);
    if (st != KVI_OK) return st;
    if (n_facts < 0 || (n_facts > 0 && !fact_len) || !sizes_out)
        return fail(KVI_ERR_INVALID_ARG, "n_facts < 0, fact_len or sizes_out NULL");
    int64_t run = 0;
    for (int64_t i = 0; i < n_facts; ++i) {
        if (fact_len[i] < 0) return fail(KVI_ERR_INVALID_ARG, "fact_len[%lld] < 0", (long long)i);
        if (token_offsets_out) token_offsets_out[i] = run;
        run += fact_len[i];
    }
    if (token_offsets_out) token_offsets_out[n_facts] = run;
    sizes_out->n_tokens = run;
    sizes_out->kv_bytes = (size_t)g->layers * 2 * (size_t)run * g->kv_heads * g->head_dim * 2;
    sizes_out->emb_bytes = (size_t)n_facts * g->embed_dim * 4;
    sizes_out->offsets_bytes = (size_t)(n_facts + 1) * 8;
    return KVI_OK;
}

kvi_status kvi_prepare_rope_ex(const kvi_rope *rope, int32_t head_dim, int32_t max_position)
{
    kvi_status st = check_rope(rope);
    if (st != KVI_OK) return st;
    if (head_dim < 16 || head_dim > KVI_MAX_HEAD_DIM || head_dim % 16)
        return fail(KVI_ERR_INVALID_ARG, "head_dim=%d must be a multiple of 16 in [16, %d]",
                    head_dim, KVI_MAX_HEAD_DIM);
    if (max_position <= 0 || max_position > kMaxRopePositions)
        return fail(KVI_ERR_INVALID_ARG, "max_position=%d outside [1, 2^22]", max_position);
    if (rope->table_id && max_position > rope->table_positions)
        return fail(KVI_ERR_INVALID_ARG, "the rope table has %d rows, fewer than max_position=%d",
                    rope->table_positions, max_position);
    const float4 *t;
    int32_t n;
    return rope_get(*rope, head_dim, max_position, nullptr, &t, &n);
}

kvi_status kvi_prepare_rope(double rope_theta, int32_t head_dim, int32_t max_position)
{
    const kvi_rope r = plain_rope(rope_theta);
    return kvi_prepare_rope_ex(&r, head_dim, max_position);
}

size_t kvi_workspace_bytes(int32_t R, int64_t max_facts, int32_t k)
{
    if (R < 1 || R > kMaxRequests || max_facts < 1 || max_facts > 0x7fffffff || k < 1 ||
        k > KVI_MAX_K)
        return 0;
    return ws_layout(R, max_facts, k).total;
}

kvi_status kvi_trace_stages(const kvi_event_t *events, int32_t n_events)
{
    if (n_events == 0) {
        t_trace_n = 0;
        return KVI_OK;
    }
    if (n_events != 3 || !events || !events[0] || !events[1] || !events[2])
        return fail(KVI_ERR_INVALID_ARG, "kvi_trace_stages wants 3 events or 0");
    for (int i = 0; i < 3; ++i) t_trace[i] = reinterpret_cast<cudaEvent_t>(events[i]);
    t_trace_n = 3;
    return KVI_OK;
}

kvi_status kvi_retrieve_topk(const kvi_store_view *store, const float *d_query, int32_t k,
                             int32_t *d_ids, float *d_scores, void *d_ws, size_t ws_bytes,
                             int32_t *d_status, kvi_stream_t stream)
{
    kvi_status st = check_store(store, true, false);
    if (st != KVI_OK) return st;
    if (!d_query || !aligned(d_query, 16))
        return fail(KVI_ERR_INVALID_ARG, "query must be a 16-byte aligned device pointer");
    if (k < 1 || k > KVI_MAX_K || (int64_t)k > store->n_facts)
        return fail(KVI_ERR_INVALID_ARG, "k=%d outside [1, min(%d, n_facts=%lld)]", k, KVI_MAX_K,
                    (long long)store->n_facts);
    if (!d_ids || !d_scores) return fail(KVI_ERR_INVALID_ARG, "ids or scores is NULL");
    if (!d_status || !aligned(d_status, 4))
        return fail(KVI_ERR_INVALID_ARG, "status must be a 4-byte aligned device pointer");
    const WsLayout w = ws_layout(1, store->n_facts, k);
    if (!d_ws || !aligned(d_ws, 256) || ws_bytes < w.total)
        return fail(KVI_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned", w.total);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(d_ws);

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
    KVI_CUDA(launch_score(sp, s));

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
    KVI_CUDA(launch_select(lp, s, true));
    return KVI_OK;
}

kvi_status kvi_place(const kvi_store_view *store, const int32_t *d_ids, int32_t n, int32_t start,
                     int32_t *d_pos, int32_t *d_status, kvi_stream_t stream)
{
    kvi_status st = check_store(store, false, false);
    if (st != KVI_OK) return st;
    if (n < 1 || n > KVI_MAX_K) return fail(KVI_ERR_INVALID_ARG, "n=%d outside [1, %d]", n, KVI_MAX_K);
    if (!d_ids || !d_pos) return fail(KVI_ERR_INVALID_ARG, "ids or pos is NULL");
    if (start < 0) return fail(KVI_ERR_INVALID_ARG, "start < 0");
    PlaceParams pp{};
    pp.store = *store;
    pp.ids = d_ids;
    pp.n = n;
    pp.start = start;
    pp.pos = d_pos;
    pp.status = d_status;
    KVI_CUDA(launch_place(pp, reinterpret_cast<cudaStream_t>(stream)));
    return KVI_OK;
}

kvi_status kvi_inject_paged(const kvi_store_view *store, const int32_t *d_fact_ids,
                            const int32_t *d_start_pos, int32_t n, const int32_t *d_block_table,
                            int32_t table_len, const kvi_paged_cache *cache, double rope_theta,
                            int32_t *d_status, kvi_stream_t stream)
{
    const kvi_rope r = plain_rope(rope_theta);
    return kvi_inject_paged_ex(store, d_fact_ids, d_start_pos, n, d_block_table, table_len, cache,
                               &r, d_status, stream);
}

kvi_status kvi_inject_paged_ex(const kvi_store_view *store, const int32_t *d_fact_ids,
                               const int32_t *d_start_pos, int32_t n, const int32_t *d_block_table,
                               int32_t table_len, const kvi_paged_cache *cache, const kvi_rope *rope,
                               int32_t *d_status, kvi_stream_t stream)
{
    kvi_status st = check_store(store, false, true);
    if (st != KVI_OK) return st;
    if (n < 1 || n > KVI_MAX_INJECT_FACTS)
        return fail(KVI_ERR_INVALID_ARG, "n=%d outside [1, %d]", n, KVI_MAX_INJECT_FACTS);
    if (!d_fact_ids || !d_start_pos || !d_block_table)
        return fail(KVI_ERR_INVALID_ARG, "fact ids, start positions or block table is NULL");
    if (table_len < 1) return fail(KVI_ERR_INVALID_ARG, "table_len < 1");
    st = check_cache(cache, store->g);
    if (st != KVI_OK) return st;
    st = check_rope(rope);
    if (st != KVI_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float4 *table;
    int32_t positions;
    st = rope_get(*rope, store->g.head_dim,
                  clamp_rope((int64_t)table_len * cache->block_size), s, &table, &positions);
    if (st != KVI_OK) return st;

    InjectParams ip{};
    ip.store.single = *store;
    ip.store.many = nullptr;
    ip.L = store->g.layers;
    ip.H = store->g.kv_heads;
    ip.D = store->g.head_dim;
    ip.pg = piece_geom(ip.H, ip.D, cache->block_size);
    ip.fused = 0;
    ip.ids = d_fact_ids;
    ip.pos = d_start_pos;
    ip.n = n;
    ip.block_tables = d_block_table;
    ip.table_len = table_len;
    ip.num_blocks = cache->num_blocks;
    ip.block_size = cache->block_size;
    ip.rope = table;
    ip.rope_positions = positions;
    ip.pairing = rope->pairing;
    ip.status = d_status;
    for (int l = 0; l < ip.L; ++l) ip.layer_base[l] = cache->layer_base[l];
#ifdef KVI_DEBUG_CHECKS
    if (d_status) KVI_CUDA(launch_overlap_check(ip, s));
#endif
    KVI_CUDA(launch_inject(ip, s, false));
    return KVI_OK;
}

kvi_status kvi_retrieve_and_inject(const kvi_geometry *g, int32_t R, const kvi_store_view *d_stores,
                                   int64_t max_facts, const float *d_queries, int32_t k,
                                   const int32_t *d_start_pos, const int32_t *d_block_tables,
                                   const int32_t *d_table_lens, int32_t max_blocks,
                                   const kvi_paged_cache *cache, double rope_theta, int32_t *d_ids,
                                   float *d_scores, int32_t *d_pos, void *d_ws, size_t ws_bytes,
                                   int32_t *d_status, kvi_stream_t stream)
{
    const kvi_rope r = plain_rope(rope_theta);
    return kvi_retrieve_and_inject_ex(g, R, d_stores, max_facts, d_queries, k, d_start_pos,
                                      d_block_tables, d_table_lens, max_blocks, cache, &r, d_ids,
                                      d_scores, d_pos, d_ws, ws_bytes, d_status, stream);
}

kvi_status kvi_retrieve_and_inject_ex(const kvi_geometry *g, int32_t R, const kvi_store_view *d_stores,
                                      int64_t max_facts, const float *d_queries, int32_t k,
                                      const int32_t *d_start_pos, const int32_t *d_block_tables,
                                      const int32_t *d_table_lens, int32_t max_blocks,
                                      const kvi_paged_cache *cache, const kvi_rope *rope,
                                      int32_t *d_ids, float *d_scores, int32_t *d_pos, void *d_ws,
                                      size_t ws_bytes, int32_t *d_status, kvi_stream_t stream)
{
    kvi_status st = check_geometry(g);
    if (st != KVI_OK) return st;
    if (R < 1 || R > kMaxRequests) return fail(KVI_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, kMaxRequests);
    if (!d_stores || !aligned(d_stores, 8)) return fail(KVI_ERR_INVALID_ARG, "stores array is NULL or misaligned");
    if (k < 1 || k > KVI_MAX_K) return fail(KVI_ERR_INVALID_ARG, "k=%d outside [1, %d]", k, KVI_MAX_K);
    if (max_facts < k || max_facts > 0x7fffffff)
        return fail(KVI_ERR_INVALID_ARG, "max_facts=%lld outside [k, 2^31)", (long long)max_facts);
    if (!d_queries || !aligned(d_queries, 16) || (g->embed_dim * 4) % 16)
        return fail(KVI_ERR_INVALID_ARG, "queries must be 16-byte aligned rows");
    if (!d_start_pos || !d_block_tables || !d_table_lens)
        return fail(KVI_ERR_INVALID_ARG, "start positions, block tables or table lengths is NULL");
    if (max_blocks < 1) return fail(KVI_ERR_INVALID_ARG, "max_blocks < 1");
    st = check_cache(cache, *g);
    if (st != KVI_OK) return st;
    if ((int64_t)max_blocks * cache->block_size > 0x7fffffff)
        return fail(KVI_ERR_INVALID_ARG, "max_blocks * block_size must be < 2^31");
    st = check_rope(rope);
    if (st != KVI_OK) return st;
    if (!d_ids || !d_scores || !d_pos) return fail(KVI_ERR_INVALID_ARG, "ids, scores or pos is NULL");
    const WsLayout w = ws_layout(R, max_facts, k);
    if (!d_ws || !aligned(d_ws, 256) || ws_bytes < w.total)
        return fail(KVI_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned", w.total);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float4 *table;
    int32_t positions;
    st = rope_get(*rope, g->head_dim, clamp_rope((int64_t)max_blocks * cache->block_size), s,
                  &table, &positions);
    if (st != KVI_OK) return st;

    const bool trace = t_trace_n == 3;
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[0], s));
    char *ws = static_cast<char *>(d_ws);
    const PieceGeom pg = piece_geom(g->kv_heads, g->head_dim, cache->block_size);

    ScoreParams sp{};
    sp.store.many = d_stores;
    sp.queries = d_queries;
    sp.g = *g;
    sp.R = R;
    sp.k = k;
    sp.max_facts = max_facts;
    sp.keys = reinterpret_cast<uint64_t *>(ws + w.keys);
    sp.lens = reinterpret_cast<int32_t *>(ws + w.lens);
    sp.key_stride = w.key_stride;
    sp.status = d_status;
    KVI_CUDA(launch_score(sp, s));

    SelectParams lp{};
    lp.store = sp.store;
    lp.g = *g;
    lp.R = R;
    lp.k = k;
    lp.max_facts = max_facts;
    lp.key_stride = w.key_stride;
    lp.keys = sp.keys;
    lp.lens = sp.lens;
    lp.ids = d_ids;
    lp.scores = d_scores;
    lp.place = 1;
    lp.start_pos = d_start_pos;
    lp.table_lens = d_table_lens;
    lp.max_blocks = max_blocks;
    lp.block_size = cache->block_size;
    lp.pg = pg;
    lp.pos = d_pos;
    lp.slot_len = reinterpret_cast<int32_t *>(ws + w.slot_len);
    lp.pc = reinterpret_cast<int32_t *>(ws + w.pc);
    lp.npc = reinterpret_cast<int32_t *>(ws + w.npc);
    lp.rows = reinterpret_cast<int64_t *>(ws + w.rows);
    lp.work = reinterpret_cast<unsigned long long *>(ws + w.work);
    lp.status = d_status;
    KVI_CUDA(launch_select(lp, s, true));
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[1], s));

    InjectParams ip{};
    ip.store.many = d_stores;
    ip.L = g->layers;
    ip.H = g->kv_heads;
    ip.D = g->head_dim;
    ip.pg = pg;
    ip.fused = 1;
    ip.ids = d_ids;
    ip.pos = d_pos;
    ip.R = R;
    ip.k = k;
    ip.slot_len = lp.slot_len;
    ip.pc = lp.pc;
    ip.npc = lp.npc;
    ip.rows = lp.rows;
    ip.work = lp.work;
    ip.block_tables = d_block_tables;
    ip.table_lens = d_table_lens;
    ip.max_blocks = max_blocks;
    ip.num_blocks = cache->num_blocks;
    ip.block_size = cache->block_size;
    ip.rope = table;
    ip.rope_positions = positions;
    ip.pairing = rope->pairing;
    ip.status = d_status;
    for (int l = 0; l < ip.L; ++l) ip.layer_base[l] = cache->layer_base[l];
    KVI_CUDA(launch_inject(ip, s, !trace));
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[2], s));
    return KVI_OK;
}

}  // extern "C"

struct kvi_plan_s {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

extern "C" {

kvi_status kvi_plan_create_fused(kvi_plan *plan, const kvi_geometry *g, int32_t R,
                                 const kvi_store_view *d_stores, int64_t max_facts,
                                 const float *d_queries, int32_t k, const int32_t *d_start_pos,
                                 const int32_t *d_block_tables, const int32_t *d_table_lens,
                                 int32_t max_blocks, const kvi_paged_cache *cache, const kvi_rope *rope,
                                 int32_t *d_ids, float *d_scores, int32_t *d_pos, void *d_ws,
                                 size_t ws_bytes, int32_t *d_status)
{
    return kvi_plan_create_fused_io(plan, g, R, d_stores, max_facts, d_queries, k, d_start_pos,
                                    d_block_tables, d_table_lens, max_blocks, cache, rope, d_ids, d_scores,
                                    d_pos, d_ws, ws_bytes, d_status, nullptr, nullptr, 0, nullptr, nullptr,
                                    0);
}

kvi_status kvi_plan_create_fused_io(kvi_plan *plan, const kvi_geometry *g, int32_t R,
                                    const kvi_store_view *d_stores, int64_t max_facts,
                                    const float *d_queries, int32_t k, const int32_t *d_start_pos,
                                    const int32_t *d_block_tables, const int32_t *d_table_lens,
                                    int32_t max_blocks, const kvi_paged_cache *cache, const kvi_rope *rope,
                                    int32_t *d_ids, float *d_scores, int32_t *d_pos, void *d_ws,
                                    size_t ws_bytes, int32_t *d_status, const void *h_in, void *d_in,
                                    size_t in_bytes, const void *d_out, void *h_out, size_t out_bytes)
{
    if (!plan) return fail(KVI_ERR_INVALID_ARG, "plan is NULL");
    if ((in_bytes && (!h_in || !d_in)) || (out_bytes && (!d_out || !h_out)))
        return fail(KVI_ERR_INVALID_ARG, "a request copy needs both of its pointers");
    *plan = nullptr;
    if (t_trace_n == 3) return fail(KVI_ERR_INVALID_ARG, "turn tracing off before recording a plan");
    kvi_status st = check_geometry(g);
    if (st != KVI_OK) return st;
    st = check_rope(rope);
    if (st != KVI_OK) return st;
    if (!cache || max_blocks < 1) return fail(KVI_ERR_INVALID_ARG, "cache is NULL or max_blocks < 1");
    // the table is built now: building it is refused while recording
    {
        const float4 *table;
        int32_t positions;
        st = rope_get(*rope, g->head_dim, clamp_rope((int64_t)max_blocks * cache->block_size), nullptr,
                      &table, &positions);
        if (st != KVI_OK) return st;
    }
    // kernel attributes are set once per device, outside the recording
    KVI_CUDA(prepare_retrieval_kernels());
    KVI_CUDA(prepare_inject_kernel());
    cudaStream_t s = nullptr;
    KVI_CUDA(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) {
        cudaStreamDestroy(s);
        return fail(KVI_ERR_CUDA, "cudaStreamBeginCapture: %s", cudaGetErrorString(e));
    }
    if (in_bytes) {
        e = cudaMemcpyAsync(d_in, h_in, in_bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) st = fail(KVI_ERR_CUDA, "request input copy: %s", cudaGetErrorString(e));
    }
    if (st == KVI_OK)
        st = kvi_retrieve_and_inject_ex(g, R, d_stores, max_facts, d_queries, k, d_start_pos,
                                        d_block_tables, d_table_lens, max_blocks, cache, rope, d_ids,
                                        d_scores, d_pos, d_ws, ws_bytes, d_status,
                                        reinterpret_cast<kvi_stream_t>(s));
    if (st == KVI_OK && out_bytes) {
        e = cudaMemcpyAsync(h_out, d_out, out_bytes, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) st = fail(KVI_ERR_CUDA, "request output copy: %s", cudaGetErrorString(e));
    }
    e = cudaStreamEndCapture(s, &graph);
    cudaStreamDestroy(s);
    if (st != KVI_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    if (e != cudaSuccess) return fail(KVI_ERR_CUDA, "cudaStreamEndCapture: %s", cudaGetErrorString(e));
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    if (e != cudaSuccess) {
        cudaGraphDestroy(graph);
        return fail(KVI_ERR_CUDA, "cudaGraphInstantiate: %s", cudaGetErrorString(e));
    }
    *plan = new kvi_plan_s{graph, exec};
    return KVI_OK;
}

kvi_status kvi_plan_launch(kvi_plan plan, kvi_stream_t stream)
{
    if (!plan) return fail(KVI_ERR_INVALID_ARG, "plan is NULL");
    KVI_CUDA(cudaGraphLaunch(plan->exec, reinterpret_cast<cudaStream_t>(stream)));
    return KVI_OK;
}

kvi_status kvi_plan_destroy(kvi_plan plan)
{
    if (!plan) return KVI_OK;
    const cudaError_t a = cudaGraphExecDestroy(plan->exec);
    const cudaError_t b = cudaGraphDestroy(plan->graph);
    delete plan;
    if (a != cudaSuccess) return fail(KVI_ERR_CUDA, "cudaGraphExecDestroy: %s", cudaGetErrorString(a));
    if (b != cudaSuccess) return fail(KVI_ERR_CUDA, "cudaGraphDestroy: %s", cudaGetErrorString(b));
    return KVI_OK;
}

size_t kvi_workspace_bytes_shared(int32_t R, int64_t n_facts, int32_t k)
{
    if (R < 1 || R > KVI_MAX_SHARED_QUERIES || n_facts < 1 || n_facts > 0x7fffffff || k < 1 ||
        k > KVI_MAX_K)
        return 0;
    return shared_layout(R, n_facts, k).total;
}

}  // extern "C"

namespace {

// Checks and the three retrieval kernels of a shared-store call: tensor-core
// coarse intervals, candidates per query, their exact keys.
kvi_status shared_retrieve(const kvi_store_view *store, bool inject, int32_t R, const float *d_queries,
                           int32_t k, void *d_ws, size_t ws_bytes, int32_t *d_status, cudaStream_t s,
                           SharedWs &L)
{
    kvi_status st = check_store(store, true, inject);
    if (st != KVI_OK) return st;
    if (R < 1 || R > KVI_MAX_SHARED_QUERIES)
        return fail(KVI_ERR_INVALID_ARG, "R=%d outside [1, %d]", R, KVI_MAX_SHARED_QUERIES);
    if (!d_queries || !aligned(d_queries, 16))
        return fail(KVI_ERR_INVALID_ARG, "queries must be a 16-byte aligned device pointer");
    if (k < 1 || k > KVI_MAX_K || (int64_t)k > store->n_facts)
        return fail(KVI_ERR_INVALID_ARG, "k=%d outside [1, min(%d, n_facts=%lld)]", k, KVI_MAX_K,
                    (long long)store->n_facts);
    L = shared_layout(R, store->n_facts, k);
    if (!d_ws || !aligned(d_ws, 256) || ws_bytes < L.total)
        return fail(KVI_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned", L.total);
    char *ws = static_cast<char *>(d_ws);
    CoarseParams cp{};
    cp.N = (int32_t)store->n_facts;
    cp.R = R;
    cp.Rp = ((R + 15) / 16) * 16;
    cp.E = store->g.embed_dim;
    cp.stride = L.w.key_stride;
    cp.lo = reinterpret_cast<float *>(ws + L.lo);
    cp.hi = reinterpret_cast<float *>(ws + L.hi);
    cp.status = d_status;
    KVI_CUDA(launch_coarse(cp, store->emb, store->n_facts, d_queries, s));
    CandParams cd{};
    cd.lo = cp.lo;
    cd.hi = cp.hi;
    cd.stride = cp.stride;
    cd.N = cp.N;
    cd.R = R;
    cd.k = k;
    cd.cand = reinterpret_cast<int32_t *>(ws + L.cand);
    cd.cand_n = reinterpret_cast<int32_t *>(ws + L.cand_n);
    KVI_CUDA(launch_candidates(cd, s, true));
    RescoreParams rp{};
    rp.store = *store;
    rp.queries = d_queries;
    rp.R = R;
    rp.stride = cp.stride;
    rp.cand = cd.cand;
    rp.cand_n = cd.cand_n;
    rp.keys = reinterpret_cast<uint64_t *>(ws + L.w.keys);
    rp.lens = reinterpret_cast<int32_t *>(ws + L.w.lens);
    KVI_CUDA(launch_rescore(rp, s, true));
    return KVI_OK;
}

SelectParams shared_select_params(const kvi_store_view *store, int32_t R, int32_t k, const SharedWs &L,
                                  char *ws, int32_t *d_ids, float *d_scores)
{
    SelectParams lp{};
    lp.store.single = *store;
    lp.store.many = nullptr;
    lp.g = store->g;
    lp.R = R;
    lp.k = k;
    lp.max_facts = store->n_facts;
    lp.key_stride = L.w.key_stride;
    lp.keys = reinterpret_cast<uint64_t *>(ws + L.w.keys);
    lp.lens = reinterpret_cast<int32_t *>(ws + L.w.lens);
    lp.cand = reinterpret_cast<int32_t *>(ws + L.cand);
    lp.cand_n = reinterpret_cast<int32_t *>(ws + L.cand_n);
    lp.ids = d_ids;
    lp.scores = d_scores;
    return lp;
}

}  // namespace

extern "C" {

kvi_status kvi_retrieve_topk_shared(const kvi_store_view *store, int32_t R, const float *d_queries,
                                    int32_t k, int32_t *d_ids, float *d_scores, void *d_ws,
                                    size_t ws_bytes, int32_t *d_status, kvi_stream_t stream)
{
    if (!d_ids || !d_scores) return fail(KVI_ERR_INVALID_ARG, "ids or scores is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    SharedWs L;
    kvi_status st = shared_retrieve(store, false, R, d_queries, k, d_ws, ws_bytes, d_status, s, L);
    if (st != KVI_OK) return st;
    SelectParams lp = shared_select_params(store, R, k, L, static_cast<char *>(d_ws), d_ids, d_scores);
    lp.place = 0;
    lp.status = d_status;
    KVI_CUDA(launch_select(lp, s, true));
    return KVI_OK;
}

kvi_status kvi_retrieve_and_inject_shared(const kvi_store_view *store, int32_t R, const float *d_queries,
                                          int32_t k, const int32_t *d_start_pos,
                                          const int32_t *d_block_tables, const int32_t *d_table_lens,
                                          int32_t max_blocks, const kvi_paged_cache *cache,
                                          const kvi_rope *rope, int32_t *d_ids, float *d_scores,
                                          int32_t *d_pos, void *d_ws, size_t ws_bytes, int32_t *d_status,
                                          kvi_stream_t stream)
{
    if (!d_ids || !d_scores || !d_pos) return fail(KVI_ERR_INVALID_ARG, "ids, scores or pos is NULL");
    if (!d_start_pos || !d_block_tables || !d_table_lens)
        return fail(KVI_ERR_INVALID_ARG, "start positions, block tables or table lengths is NULL");
    if (max_blocks < 1) return fail(KVI_ERR_INVALID_ARG, "max_blocks < 1");
    if (!store) return fail(KVI_ERR_INVALID_ARG, "store is NULL");
    kvi_status st = check_cache(cache, store->g);
    if (st != KVI_OK) return st;
    if ((int64_t)max_blocks * cache->block_size > 0x7fffffff)
        return fail(KVI_ERR_INVALID_ARG, "max_blocks * block_size must be < 2^31");
    st = check_rope(rope);
    if (st != KVI_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float4 *table;
    int32_t positions;
    st = rope_get(*rope, store->g.head_dim, clamp_rope((int64_t)max_blocks * cache->block_size), s, &table,
                  &positions);
    if (st != KVI_OK) return st;
    const bool trace = t_trace_n == 3;
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[0], s));
    SharedWs L;
    st = shared_retrieve(store, true, R, d_queries, k, d_ws, ws_bytes, d_status, s, L);
    if (st != KVI_OK) return st;
    char *ws = static_cast<char *>(d_ws);
    const PieceGeom pg = piece_geom(store->g.kv_heads, store->g.head_dim, cache->block_size);
    SelectParams lp = shared_select_params(store, R, k, L, ws, d_ids, d_scores);
    lp.place = 1;
    lp.start_pos = d_start_pos;
    lp.table_lens = d_table_lens;
    lp.max_blocks = max_blocks;
    lp.block_size = cache->block_size;
    lp.pg = pg;
    lp.pos = d_pos;
    lp.slot_len = reinterpret_cast<int32_t *>(ws + L.w.slot_len);
    lp.pc = reinterpret_cast<int32_t *>(ws + L.w.pc);
    lp.npc = reinterpret_cast<int32_t *>(ws + L.w.npc);
    lp.rows = reinterpret_cast<int64_t *>(ws + L.w.rows);
    lp.work = reinterpret_cast<unsigned long long *>(ws + L.w.work);
    lp.status = d_status;
    KVI_CUDA(launch_select(lp, s, true));
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[1], s));

    InjectParams ip{};
    ip.store.single = *store;
    ip.store.many = nullptr;
    ip.L = store->g.layers;
    ip.H = store->g.kv_heads;
    ip.D = store->g.head_dim;
    ip.pg = pg;
    ip.fused = 1;
    ip.ids = d_ids;
    ip.pos = d_pos;
    ip.R = R;
    ip.k = k;
    ip.slot_len = lp.slot_len;
    ip.pc = lp.pc;
    ip.npc = lp.npc;
    ip.rows = lp.rows;
    ip.work = lp.work;
    ip.block_tables = d_block_tables;
    ip.table_lens = d_table_lens;
    ip.max_blocks = max_blocks;
    ip.num_blocks = cache->num_blocks;
    ip.block_size = cache->block_size;
    ip.rope = table;
    ip.rope_positions = positions;
    ip.pairing = rope->pairing;
    ip.status = d_status;
    for (int l = 0; l < ip.L; ++l) ip.layer_base[l] = cache->layer_base[l];
    KVI_CUDA(launch_inject(ip, s, !trace));
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[2], s));
    return KVI_OK;
}

}  // extern "C"

// ------------------------------------------------------------- graph index

namespace {

struct GraphBuildWs {
    SharedWs shared;
    size_t ids, scores, total;
};

GraphBuildWs graph_build_layout(int64_t n_facts, int32_t degree)
{
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    GraphBuildWs x{};
    const int32_t R = (int32_t)std::min<int64_t>(KVI_MAX_SHARED_QUERIES, n_facts);
    const int32_t k = degree + 1;
    x.shared = shared_layout(R, n_facts, k);
    size_t at = up(x.shared.total);
    x.ids = at;    at = up(at + (size_t)R * k * 4);
    x.scores = at; at = up(at + (size_t)R * k * 4);
    x.total = at;
    return x;
}

bool graph_build_args_ok(int64_t n_facts, int32_t degree)
{
    return n_facts >= 2 && n_facts <= 0x7fffffff && degree >= 1 && degree <= KVI_MAX_GRAPH_DEGREE &&
           (int64_t)degree < n_facts;
}


struct GraphFusedWs {
    SharedWs sel;  // the selector's regions and candidate lists (beam slots)
    size_t visited, total;
};

GraphFusedWs graph_fused_layout(int32_t R, int64_t n_facts, int32_t beam, int32_t k)
{
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    GraphFusedWs x{};
    x.sel = shared_layout(R, beam, k);
    x.visited = up(x.sel.total);
    x.total = up(x.visited + (size_t)R * (size_t)((n_facts + 31) / 32) * 4);
    return x;
}

// The argument checks kvi_graph_search and the fused graph call share.
kvi_status check_graph_search(const kvi_store_view *store, const int32_t *d_graph, int32_t degree,
                              int32_t R, const float *d_queries, const int32_t *d_seeds,
                              const kvi_graph_search_params *params, int32_t k, bool inject)
{
    kvi_status st = check_store(store, true, inject);
    if (st != KVI_OK) return st;
    if (!d_graph || !aligned(d_graph, 4)) return fail(KVI_ERR_INVALID_ARG, "graph is NULL or misaligned");
    if (degree < 1 || degree > KVI_MAX_GRAPH_DEGREE)
        return fail(KVI_ERR_INVALID_ARG, "degree=%d outside [1, %d]", degree, KVI_MAX_GRAPH_DEGREE);
    if (R < 1 || R > 65535) return fail(KVI_ERR_INVALID_ARG, "R=%d outside [1, 65535]", R);
    if (!d_queries || !aligned(d_queries, 16))
        return fail(KVI_ERR_INVALID_ARG, "queries must be a 16-byte aligned device pointer");
    if (!d_seeds || !params) return fail(KVI_ERR_INVALID_ARG, "seeds or params is NULL");
    const kvi_graph_search_params P = *params;
    if (k < 1 || P.beam < k || P.beam > KVI_MAX_GRAPH_BEAM)
        return fail(KVI_ERR_INVALID_ARG, "need 1 <= k=%d <= beam=%d <= %d", k, P.beam, KVI_MAX_GRAPH_BEAM);
    if (P.width < 1 || (int64_t)P.width * degree > KVI_MAX_GRAPH_FRONTIER)
        return fail(KVI_ERR_INVALID_ARG, "width=%d: need 1 <= width * degree <= %d", P.width,
                    KVI_MAX_GRAPH_FRONTIER);
    if (P.max_iters < 0 || P.n_seeds < 1 || P.n_seeds > KVI_MAX_GRAPH_FRONTIER)
        return fail(KVI_ERR_INVALID_ARG, "max_iters=%d < 0 or n_seeds=%d outside [1, %d]", P.max_iters,
                    P.n_seeds, KVI_MAX_GRAPH_FRONTIER);
    return KVI_OK;
}

GraphSearchParams graph_params(const kvi_store_view *store, const int32_t *d_graph, int32_t degree, int32_t R,
                               const float *d_queries, const int32_t *d_seeds,
                               const kvi_graph_search_params &P, int32_t k, uint32_t *visited,
                               int32_t *d_status)
{
    GraphSearchParams gp{};
    gp.emb = store->emb;
    gp.N = store->n_facts;
    gp.E = store->g.embed_dim;
    gp.graph = d_graph;
    gp.degree = degree;
    gp.queries = d_queries;
    gp.seeds = d_seeds;
    gp.R = R;
    gp.n_seeds = P.n_seeds;
    gp.beam = P.beam;
    gp.width = P.width;
    gp.max_iters = P.max_iters;
    gp.k = k;
    gp.visited = visited;
    gp.vis_words = (store->n_facts + 31) / 32;
    gp.status = d_status;
    gp.fact_start = store->fact_start;
    gp.fact_len = store->fact_len;
    gp.n_tokens = store->n_tokens;
    return gp;
}

}  // namespace

extern "C" {

size_t kvi_graph_build_workspace_bytes(int64_t n_facts, int32_t degree)
{
    if (!graph_build_args_ok(n_facts, degree)) return 0;
    return graph_build_layout(n_facts, degree).total;
}

kvi_status kvi_graph_build(const kvi_store_view *store, int32_t degree, int32_t *d_graph, void *d_ws,
                           size_t ws_bytes, int32_t *d_status, kvi_stream_t stream)
{
    kvi_status st = check_store(store, true, false);
    if (st != KVI_OK) return st;
    const int64_t N = store->n_facts;
    if (!graph_build_args_ok(N, degree))
        return fail(KVI_ERR_INVALID_ARG, "degree=%d outside [1, min(%d, n_facts - 1 = %lld)]", degree,
                    KVI_MAX_GRAPH_DEGREE, (long long)(N - 1));
    if (!d_graph || !aligned(d_graph, 4)) return fail(KVI_ERR_INVALID_ARG, "graph is NULL or misaligned");
    const GraphBuildWs W = graph_build_layout(N, degree);
    if (!d_ws || !aligned(d_ws, 256) || ws_bytes < W.total)
        return fail(KVI_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned", W.total);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(d_ws);
    int32_t *ids = reinterpret_cast<int32_t *>(ws + W.ids);
    float *scores = reinterpret_cast<float *>(ws + W.scores);
    const int32_t k = degree + 1;
    const int64_t E = store->g.embed_dim;
    for (int64_t i0 = 0; i0 < N; i0 += KVI_MAX_SHARED_QUERIES) {
        const int32_t R = (int32_t)std::min<int64_t>(KVI_MAX_SHARED_QUERIES, N - i0);
        SharedWs L;
        st = shared_retrieve(store, false, R, store->emb + i0 * E, k, d_ws, W.shared.total, d_status, s, L);
        if (st != KVI_OK) return st;
        SelectParams lp = shared_select_params(store, R, k, L, ws, ids, scores);
        lp.place = 0;
        lp.status = d_status;
        KVI_CUDA(launch_select(lp, s, true));
        GraphRowsParams gp{ids, i0, R, degree, d_graph};
        KVI_CUDA(launch_graph_rows(gp, s));
    }
    return KVI_OK;
}

size_t kvi_graph_search_workspace_bytes(int32_t R, int64_t n_facts)
{
    if (R < 1 || R > 65535 || n_facts < 1 || n_facts > 0x7fffffff) return 0;
    return (size_t)R * (size_t)((n_facts + 31) / 32) * 4;
}

kvi_status kvi_graph_search(const kvi_store_view *store, const int32_t *d_graph, int32_t degree, int32_t R,
                            const float *d_queries, const int32_t *d_seeds,
                            const kvi_graph_search_params *params, int32_t k, int32_t *d_ids,
                            float *d_scores, int32_t *d_count, int32_t *d_stats, void *d_ws,
                            size_t ws_bytes, int32_t *d_status, kvi_stream_t stream)
{
    kvi_status st = check_graph_search(store, d_graph, degree, R, d_queries, d_seeds, params, k, false);
    if (st != KVI_OK) return st;
    if (!d_ids || !d_scores) return fail(KVI_ERR_INVALID_ARG, "ids or scores is NULL");
    const size_t need = kvi_graph_search_workspace_bytes(R, store->n_facts);
    if (!d_ws || !aligned(d_ws, 256) || ws_bytes < need)
        return fail(KVI_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned", need);
    GraphSearchParams gp = graph_params(store, d_graph, degree, R, d_queries, d_seeds, *params, k,
                                        static_cast<uint32_t *>(d_ws), d_status);
    gp.ids = d_ids;
    gp.scores = d_scores;
    gp.count = d_count;
    gp.stats = d_stats;
    KVI_CUDA(launch_graph_search(gp, reinterpret_cast<cudaStream_t>(stream)));
    return KVI_OK;
}

}  // extern "C"


extern "C" {

size_t kvi_graph_retrieve_and_inject_workspace_bytes(int32_t R, int64_t n_facts, int32_t beam, int32_t k)
{
    if (R < 1 || R > KVI_MAX_REQUESTS || n_facts < 1 || n_facts > 0x7fffffff || k < 1 || beam < k ||
        beam > KVI_MAX_GRAPH_BEAM)
        return 0;
    return graph_fused_layout(R, n_facts, beam, k).total;
}

kvi_status kvi_graph_retrieve_and_inject(const kvi_store_view *store, const int32_t *d_graph, int32_t degree,
                                         int32_t R, const float *d_queries, const int32_t *d_seeds,
                                         const kvi_graph_search_params *params, int32_t k,
                                         const int32_t *d_start_pos, const int32_t *d_block_tables,
                                         const int32_t *d_table_lens, int32_t max_blocks,
                                         const kvi_paged_cache *cache, const kvi_rope *rope, int32_t *d_ids,
                                         float *d_scores, int32_t *d_pos, void *d_ws, size_t ws_bytes,
                                         int32_t *d_status, kvi_stream_t stream)
{
    kvi_status st = check_graph_search(store, d_graph, degree, R, d_queries, d_seeds, params, k, true);
    if (st != KVI_OK) return st;
    if (R > KVI_MAX_REQUESTS) return fail(KVI_ERR_INVALID_ARG, "R=%d > %d", R, KVI_MAX_REQUESTS);
    if (!d_ids || !d_scores || !d_pos) return fail(KVI_ERR_INVALID_ARG, "ids, scores or pos is NULL");
    if (!d_start_pos || !d_block_tables || !d_table_lens)
        return fail(KVI_ERR_INVALID_ARG, "start positions, block tables or table lengths is NULL");
    if (max_blocks < 1) return fail(KVI_ERR_INVALID_ARG, "max_blocks < 1");
    st = check_cache(cache, store->g);
    if (st != KVI_OK) return st;
    if ((int64_t)max_blocks * cache->block_size > 0x7fffffff)
        return fail(KVI_ERR_INVALID_ARG, "max_blocks * block_size must be < 2^31");
    st = check_rope(rope);
    if (st != KVI_OK) return st;
    const GraphFusedWs W = graph_fused_layout(R, store->n_facts, params->beam, k);
    if (!d_ws || !aligned(d_ws, 256) || ws_bytes < W.total)
        return fail(KVI_ERR_INVALID_ARG, "workspace needs %zu bytes, 256-byte aligned", W.total);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const float4 *table;
    int32_t positions;
    st = rope_get(*rope, store->g.head_dim, clamp_rope((int64_t)max_blocks * cache->block_size), s, &table,
                  &positions);
    if (st != KVI_OK) return st;
    const bool trace = t_trace_n == 3;
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[0], s));
    char *ws = static_cast<char *>(d_ws);
    const SharedWs &L = W.sel;
    GraphSearchParams gp = graph_params(store, d_graph, degree, R, d_queries, d_seeds, *params, k,
                                        reinterpret_cast<uint32_t *>(ws + W.visited), d_status);
    gp.cand_ids = reinterpret_cast<int32_t *>(ws + L.cand);
    gp.cand_keys = reinterpret_cast<uint64_t *>(ws + L.w.keys);
    gp.cand_lens = reinterpret_cast<int32_t *>(ws + L.w.lens);
    gp.cand_n = reinterpret_cast<int32_t *>(ws + L.cand_n);
    gp.cand_stride = L.w.key_stride;
    KVI_CUDA(launch_graph_search(gp, s));

    const PieceGeom pg = piece_geom(store->g.kv_heads, store->g.head_dim, cache->block_size);
    SelectParams lp = shared_select_params(store, R, k, L, ws, d_ids, d_scores);
    lp.place = 1;
    lp.start_pos = d_start_pos;
    lp.table_lens = d_table_lens;
    lp.max_blocks = max_blocks;
    lp.block_size = cache->block_size;
    lp.pg = pg;
    lp.pos = d_pos;
    lp.slot_len = reinterpret_cast<int32_t *>(ws + L.w.slot_len);
    lp.pc = reinterpret_cast<int32_t *>(ws + L.w.pc);
    lp.npc = reinterpret_cast<int32_t *>(ws + L.w.npc);
    lp.rows = reinterpret_cast<int64_t *>(ws + L.w.rows);
    lp.work = reinterpret_cast<unsigned long long *>(ws + L.w.work);
    lp.status = d_status;
    KVI_CUDA(launch_select(lp, s, true));
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[1], s));

    InjectParams ip{};
    ip.store.single = *store;
    ip.store.many = nullptr;
    ip.L = store->g.layers;
    ip.H = store->g.kv_heads;
    ip.D = store->g.head_dim;
    ip.pg = pg;
    ip.fused = 1;
    ip.ids = d_ids;
    ip.pos = d_pos;
    ip.R = R;
    ip.k = k;
    ip.slot_len = lp.slot_len;
    ip.pc = lp.pc;
    ip.npc = lp.npc;
    ip.rows = lp.rows;
    ip.work = lp.work;
    ip.block_tables = d_block_tables;
    ip.table_lens = d_table_lens;
    ip.max_blocks = max_blocks;
    ip.num_blocks = cache->num_blocks;
    ip.block_size = cache->block_size;
    ip.rope = table;
    ip.rope_positions = positions;
    ip.pairing = rope->pairing;
    ip.status = d_status;
    for (int l = 0; l < ip.L; ++l) ip.layer_base[l] = cache->layer_base[l];
    KVI_CUDA(launch_inject(ip, s, !trace));
    if (trace) KVI_CUDA(cudaEventRecord(t_trace[2], s));
    return KVI_OK;
}

}  // extern "C"

extern "C" {

kvi_status kvi_selftest_bounded_wait(uint64_t limit_ns, int32_t *d_status, int64_t *d_elapsed_ns,
                                     kvi_stream_t stream)
{
    if (!d_status) return fail(KVI_ERR_INVALID_ARG, "status is NULL");
    if (limit_ns < 1000 || limit_ns > 1000000000ull)
        return fail(KVI_ERR_INVALID_ARG, "limit_ns=%llu outside [1e3, 1e9]", (unsigned long long)limit_ns);
    KVI_CUDA(launch_bounded_wait(limit_ns, d_status, d_elapsed_ns, reinterpret_cast<cudaStream_t>(stream)));
    return KVI_OK;
}

kvi_status kvi_selftest_stream_read(const void *src, size_t bytes, int32_t ctas_per_sm, uint64_t *d_sum,
                                    kvi_stream_t stream)
{
    if (!src || !d_sum || !aligned(src, 16) || bytes % 16 || !aligned(d_sum, 8))
        return fail(KVI_ERR_INVALID_ARG, "src (16-byte aligned), bytes (multiple of 16) and sum are required");
    if (ctas_per_sm < 1 || ctas_per_sm > 8)
        return fail(KVI_ERR_INVALID_ARG, "ctas_per_sm=%d outside [1, 8]", ctas_per_sm);
    KVI_CUDA(launch_stream_read(src, bytes, ctas_per_sm, d_sum, reinterpret_cast<cudaStream_t>(stream)));
    return KVI_OK;
}

}  // extern "C"

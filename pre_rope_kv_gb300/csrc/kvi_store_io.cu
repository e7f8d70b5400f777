// Store files: a fact store (fact extents, retrieval embeddings, pre-RoPE
// K/V) written to disk and read back into HBM or pinned host memory.
//
// "InferScale: GPU-Native KV Injection for Personalized LLM Serving" encodes
// a user's memory facts offline into a long-lived store that the serving
// path reads (review Summary: facts are encoded offline; the KV store may be
// offloaded to host DRAM).  The file format is documented in kvi.h next to
// the entry points; this file is host code only (blocking CUDA copies
// through a pinned bounce buffer, stdio for the file).
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <unistd.h>

#include <cuda_runtime.h>

#include "kvi_internal.cuh"

static_assert(__BYTE_ORDER__ == __ORDER_LITTLE_ENDIAN__, "the store file is little-endian");

namespace kvi {
namespace {

constexpr char kMagic[8] = {'K', 'V', 'I', 'S', 'T', 'O', 'R', 'E'};
constexpr uint32_t kVersion = 1;
constexpr uint32_t kHeaderBytes = 128;
constexpr uint64_t kSectionAlign = 4096;
constexpr uint64_t kFnvBasis = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;
constexpr size_t kChunk = size_t(32) << 20;  // bounce buffer (a multiple of 32 bytes)

kvi_status io_fail(kvi_status s, const std::string &msg) { return set_error(s, msg.c_str()); }

uint64_t round_up(uint64_t x) { return (x + kSectionAlign - 1) / kSectionAlign * kSectionAlign; }

uint64_t fnv1a(uint64_t h, const void *data, size_t n)
{
    const uint8_t *p = static_cast<const uint8_t *>(data);
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= kFnvPrime;
    }
    return h;
}

uint64_t rotl(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }

// Four-lane word hash of the payload (word i goes to lane i mod 4).
struct PayloadHash {
    uint64_t h[4] = {kFnvBasis, kFnvBasis + 1, kFnvBasis + 2, kFnvBasis + 3};
    uint64_t words = 0;

    void add(const void *data, size_t n)  // n is a multiple of 8
    {
        const uint8_t *p = static_cast<const uint8_t *>(data);
        size_t i = 0;
        for (; i < n && (words & 3); i += 8) one(p + i);
        for (; i + 32 <= n; i += 32) {
            uint64_t w[4];
            std::memcpy(w, p + i, 32);
            h[0] = (h[0] ^ w[0]) * kFnvPrime;
            h[1] = (h[1] ^ w[1]) * kFnvPrime;
            h[2] = (h[2] ^ w[2]) * kFnvPrime;
            h[3] = (h[3] ^ w[3]) * kFnvPrime;
            words += 4;
        }
        for (; i < n; i += 8) one(p + i);
    }
    void one(const uint8_t *p)
    {
        uint64_t w;
        std::memcpy(&w, p, 8);
        const int j = (int)(words & 3);
        h[j] = (h[j] ^ w) * kFnvPrime;
        ++words;
    }
    uint64_t value() const { return h[0] ^ rotl(h[1], 16) ^ rotl(h[2], 32) ^ rotl(h[3], 48); }
};

// The section layout a header must describe (fixed by the sizes).
struct Layout {
    uint64_t start_off, len_off, emb_off, kv_off, file_bytes;
    uint64_t emb_bytes, kv_bytes;
};

Layout layout_of(const kvi_geometry &g, int64_t n, int64_t t)
{
    Layout o;
    o.emb_bytes = (uint64_t)n * (uint64_t)g.embed_dim * 4u;
    o.kv_bytes = (uint64_t)g.layers * 2u * (uint64_t)t * (uint64_t)g.kv_heads * (uint64_t)g.head_dim * 2u;
    o.start_off = round_up(kHeaderBytes);
    o.len_off = round_up(o.start_off + 8u * (uint64_t)n);
    o.emb_off = round_up(o.len_off + 4u * (uint64_t)n);
    o.kv_off = round_up(o.emb_off + o.emb_bytes);
    o.file_bytes = o.kv_off + o.kv_bytes;
    return o;
}

template <typename T>
void put(uint8_t *h, size_t at, T v) { std::memcpy(h + at, &v, sizeof v); }
template <typename T>
T get(const uint8_t *h, size_t at)
{
    T v;
    std::memcpy(&v, h + at, sizeof v);
    return v;
}

struct File {
    FILE *f = nullptr;
    ~File()
    {
        if (f) fclose(f);
    }
};

struct Pinned {
    uint8_t *p = nullptr;
    ~Pinned()
    {
        if (p) cudaFreeHost(p);
    }
};

bool write_zeros(FILE *f, uint64_t n)
{
    static const uint8_t zero[4096] = {};
    while (n) {
        const size_t c = (size_t)(n < sizeof zero ? n : sizeof zero);
        if (fwrite(zero, 1, c, f) != c) return false;
        n -= c;
    }
    return true;
}

bool pad_to(FILE *f, uint64_t &at, uint64_t target)
{
    if (!write_zeros(f, target - at)) return false;
    at = target;
    return true;
}

// Header of an open file: checked against the format, its own hash, the
// canonical layout and the file's size.
struct Header {
    kvi_geometry g;
    int64_t n, t;
    Layout lay;
    uint64_t extents_hash, payload_hash;
};

kvi_status read_header(FILE *f, const char *path, Header *out)
{
    uint8_t h[kHeaderBytes];
    if (fread(h, 1, kHeaderBytes, f) != kHeaderBytes)
        return io_fail(KVI_ERR_IO, std::string(path) + ": shorter than a store file header");
    if (std::memcmp(h, kMagic, 8) != 0) return io_fail(KVI_ERR_IO, std::string(path) + ": not a store file");
    if (get<uint32_t>(h, 8) != kVersion || get<uint32_t>(h, 12) != kHeaderBytes)
        return io_fail(KVI_ERR_IO, std::string(path) + ": unsupported store file version");
    if (fnv1a(kFnvBasis, h, 104) != get<uint64_t>(h, 104))
        return io_fail(KVI_ERR_IO, std::string(path) + ": header hash mismatch");
    Header o;
    o.g.layers = get<int32_t>(h, 16);
    o.g.kv_heads = get<int32_t>(h, 20);
    o.g.head_dim = get<int32_t>(h, 24);
    o.g.embed_dim = get<int32_t>(h, 28);
    o.n = get<int64_t>(h, 32);
    o.t = get<int64_t>(h, 40);
    if (check_store_geometry(&o.g) != KVI_OK)
        return io_fail(KVI_ERR_IO, std::string(path) + ": geometry outside the library's compile-time limits");
    if (o.n < 1 || o.n > 0x7fffffff || o.t < 0 || o.t > (int64_t(1) << 40))
        return io_fail(KVI_ERR_IO, std::string(path) + ": fact or token count out of range");
    o.lay = layout_of(o.g, o.n, o.t);
    const uint64_t offs[5] = {o.lay.start_off, o.lay.len_off, o.lay.emb_off, o.lay.kv_off, o.lay.file_bytes};
    for (int i = 0; i < 5; ++i)
        if (get<uint64_t>(h, 48 + 8 * i) != offs[i])
            return io_fail(KVI_ERR_IO, std::string(path) + ": section offsets do not match the sizes");
    for (int i = 112; i < 128; ++i)
        if (h[i]) return io_fail(KVI_ERR_IO, std::string(path) + ": reserved header bytes are not zero");
    o.extents_hash = get<uint64_t>(h, 88);
    o.payload_hash = get<uint64_t>(h, 96);
    if (fseeko(f, 0, SEEK_END) != 0 || (uint64_t)ftello(f) != o.lay.file_bytes)
        return io_fail(KVI_ERR_IO, std::string(path) + ": file size does not match the header");
    *out = o;
    return KVI_OK;
}

kvi_status cuda_fail(const char *what, cudaError_t e)
{
    return io_fail(KVI_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

}  // namespace
}  // namespace kvi

using namespace kvi;

kvi_status kvi_store_save(const char *path, const kvi_store_view *s)
{
    if (!path || !*path) return io_fail(KVI_ERR_INVALID_ARG, "path is NULL or empty");
    kvi_status st = check_full_store(s);
    if (st != KVI_OK) return st;
    if (s->flags & ~KVI_STORE_KV_HOST) return io_fail(KVI_ERR_INVALID_ARG, "unknown store flags");
    const int64_t n = s->n_facts, t = s->n_tokens;
    const Layout lay = layout_of(s->g, n, t);

    std::vector<int64_t> start((size_t)n);
    std::vector<int32_t> len((size_t)n);
    cudaError_t ce = cudaMemcpy(start.data(), s->fact_start, (size_t)n * 8, cudaMemcpyDefault);
    if (ce == cudaSuccess) ce = cudaMemcpy(len.data(), s->fact_len, (size_t)n * 4, cudaMemcpyDefault);
    if (ce != cudaSuccess) return cuda_fail("reading the fact extents", ce);
    uint64_t extents = fnv1a(kFnvBasis, start.data(), (size_t)n * 8);
    extents = fnv1a(extents, len.data(), (size_t)n * 4);

    Pinned bounce;
    ce = cudaMallocHost(reinterpret_cast<void **>(&bounce.p), kChunk);
    if (ce != cudaSuccess) return cuda_fail("cudaMallocHost (bounce buffer)", ce);

    const std::string tmp = std::string(path) + ".partial." + std::to_string((long long)getpid());
    auto io_error = [&](const char *what) {
        std::remove(tmp.c_str());
        return io_fail(KVI_ERR_IO, std::string(path) + ": " + what);
    };
    PayloadHash ph;
    {
        File f;
        f.f = fopen(tmp.c_str(), "wb");
        if (!f.f) return io_fail(KVI_ERR_IO, std::string(path) + ": cannot create the file");
        uint64_t at = 0;
        // the header is written last, once the payload hash is known
        if (!pad_to(f.f, at, lay.start_off)) return io_error("write failed");
        if (fwrite(start.data(), 8, (size_t)n, f.f) != (size_t)n) return io_error("write failed");
        at += 8u * (uint64_t)n;
        if (!pad_to(f.f, at, lay.len_off)) return io_error("write failed");
        if (fwrite(len.data(), 4, (size_t)n, f.f) != (size_t)n) return io_error("write failed");
        at += 4u * (uint64_t)n;
        if (!pad_to(f.f, at, lay.emb_off)) return io_error("write failed");
        // payload: emb (device), then kv (device or host)
        struct Part {
            const uint8_t *src;
            uint64_t bytes;
            bool host;
        };
        const Part parts[2] = {{reinterpret_cast<const uint8_t *>(s->emb), lay.emb_bytes, false},
                               {static_cast<const uint8_t *>(s->kv), lay.kv_bytes,
                                (s->flags & KVI_STORE_KV_HOST) != 0}};
        for (int pi = 0; pi < 2; ++pi) {
            if (pi == 1 && !pad_to(f.f, at, lay.kv_off)) return io_error("write failed");
            const Part &pt = parts[pi];
            for (uint64_t o = 0; o < pt.bytes; o += kChunk) {
                const size_t c = (size_t)((pt.bytes - o) < kChunk ? (pt.bytes - o) : kChunk);
                const uint8_t *buf = pt.src + o;
                if (!pt.host) {
                    ce = cudaMemcpy(bounce.p, pt.src + o, c, cudaMemcpyDefault);
                    if (ce != cudaSuccess) {
                        std::remove(tmp.c_str());
                        return cuda_fail("reading the store", ce);
                    }
                    buf = bounce.p;
                }
                ph.add(buf, c);
                if (fwrite(buf, 1, c, f.f) != c) return io_error("write failed");
                at += c;
            }
        }
        uint8_t h[kHeaderBytes] = {};
        std::memcpy(h, kMagic, 8);
        put<uint32_t>(h, 8, kVersion);
        put<uint32_t>(h, 12, kHeaderBytes);
        put<int32_t>(h, 16, s->g.layers);
        put<int32_t>(h, 20, s->g.kv_heads);
        put<int32_t>(h, 24, s->g.head_dim);
        put<int32_t>(h, 28, s->g.embed_dim);
        put<int64_t>(h, 32, n);
        put<int64_t>(h, 40, t);
        put<uint64_t>(h, 48, lay.start_off);
        put<uint64_t>(h, 56, lay.len_off);
        put<uint64_t>(h, 64, lay.emb_off);
        put<uint64_t>(h, 72, lay.kv_off);
        put<uint64_t>(h, 80, lay.file_bytes);
        put<uint64_t>(h, 88, extents);
        put<uint64_t>(h, 96, ph.value());
        put<uint64_t>(h, 104, fnv1a(kFnvBasis, h, 104));
        if (fseeko(f.f, 0, SEEK_SET) != 0 || fwrite(h, 1, kHeaderBytes, f.f) != kHeaderBytes)
            return io_error("write failed");
        if (fflush(f.f) != 0) return io_error("write failed");
        const int rc = fclose(f.f);
        f.f = nullptr;
        if (rc != 0) return io_error("write failed");
    }
    if (std::rename(tmp.c_str(), path) != 0) return io_error("cannot replace the file");
    return KVI_OK;
}

kvi_status kvi_store_file_info_read(const char *path, kvi_store_file_info *info)
{
    if (!path || !info) return io_fail(KVI_ERR_INVALID_ARG, "path or info is NULL");
    File f;
    f.f = fopen(path, "rb");
    if (!f.f) return io_fail(KVI_ERR_IO, std::string(path) + ": cannot open the file");
    Header h;
    kvi_status st = read_header(f.f, path, &h);
    if (st != KVI_OK) return st;
    info->g = h.g;
    info->n_facts = h.n;
    info->n_tokens = h.t;
    info->kv_bytes = (size_t)h.lay.kv_bytes;
    info->emb_bytes = (size_t)h.lay.emb_bytes;
    return KVI_OK;
}

kvi_status kvi_store_load(const char *path, void *kv, float *emb, int64_t *fact_start, int32_t *fact_len,
                          uint32_t flags)
{
    if (!path || !emb || !fact_start || !fact_len)
        return io_fail(KVI_ERR_INVALID_ARG, "path, emb, fact_start or fact_len is NULL");
    if (flags & ~KVI_STORE_KV_HOST) return io_fail(KVI_ERR_INVALID_ARG, "unknown store flags");
    if (reinterpret_cast<uintptr_t>(emb) % 16 || reinterpret_cast<uintptr_t>(fact_start) % 8 ||
        reinterpret_cast<uintptr_t>(fact_len) % 4 || reinterpret_cast<uintptr_t>(kv) % 16)
        return io_fail(KVI_ERR_INVALID_ARG, "kv and emb must be 16-byte aligned, fact_start 8, fact_len 4");
    File f;
    f.f = fopen(path, "rb");
    if (!f.f) return io_fail(KVI_ERR_IO, std::string(path) + ": cannot open the file");
    Header h;
    kvi_status st = read_header(f.f, path, &h);
    if (st != KVI_OK) return st;
    if (!kv && h.lay.kv_bytes) return io_fail(KVI_ERR_INVALID_ARG, "kv is NULL");
    const std::string p(path);

    std::vector<int64_t> start((size_t)h.n);
    std::vector<int32_t> len((size_t)h.n);
    if (fseeko(f.f, (off_t)h.lay.start_off, SEEK_SET) != 0 ||
        fread(start.data(), 8, (size_t)h.n, f.f) != (size_t)h.n ||
        fseeko(f.f, (off_t)h.lay.len_off, SEEK_SET) != 0 || fread(len.data(), 4, (size_t)h.n, f.f) != (size_t)h.n)
        return io_fail(KVI_ERR_IO, p + ": read failed (fact extents)");
    uint64_t extents = fnv1a(kFnvBasis, start.data(), (size_t)h.n * 8);
    extents = fnv1a(extents, len.data(), (size_t)h.n * 4);
    if (extents != h.extents_hash) return io_fail(KVI_ERR_IO, p + ": fact extents hash mismatch");
    for (int64_t i = 0; i < h.n; ++i)
        if (start[(size_t)i] < 0 || len[(size_t)i] < 0 || start[(size_t)i] + len[(size_t)i] > h.t)
            return io_fail(KVI_ERR_IO, p + ": fact " + std::to_string((long long)i) + " lies outside the store");

    Pinned bounce;
    cudaError_t ce = cudaMallocHost(reinterpret_cast<void **>(&bounce.p), kChunk);
    if (ce != cudaSuccess) return cuda_fail("cudaMallocHost (bounce buffer)", ce);
    ce = cudaMemcpy(fact_start, start.data(), (size_t)h.n * 8, cudaMemcpyDefault);
    if (ce == cudaSuccess) ce = cudaMemcpy(fact_len, len.data(), (size_t)h.n * 4, cudaMemcpyDefault);
    if (ce != cudaSuccess) return cuda_fail("writing the fact extents", ce);

    PayloadHash ph;
    struct Part {
        uint8_t *dst;
        uint64_t off, bytes;
        bool host;
    };
    const Part parts[2] = {{reinterpret_cast<uint8_t *>(emb), h.lay.emb_off, h.lay.emb_bytes, false},
                           {static_cast<uint8_t *>(kv), h.lay.kv_off, h.lay.kv_bytes,
                            (flags & KVI_STORE_KV_HOST) != 0}};
    for (const Part &pt : parts) {
        if (fseeko(f.f, (off_t)pt.off, SEEK_SET) != 0) return io_fail(KVI_ERR_IO, p + ": seek failed");
        for (uint64_t o = 0; o < pt.bytes; o += kChunk) {
            const size_t c = (size_t)((pt.bytes - o) < kChunk ? (pt.bytes - o) : kChunk);
            uint8_t *buf = pt.host ? pt.dst + o : bounce.p;
            if (fread(buf, 1, c, f.f) != c) return io_fail(KVI_ERR_IO, p + ": read failed (payload)");
            ph.add(buf, c);
            if (!pt.host) {
                ce = cudaMemcpy(pt.dst + o, bounce.p, c, cudaMemcpyDefault);
                if (ce != cudaSuccess) return cuda_fail("writing the store", ce);
            }
        }
    }
    if (ph.value() != h.payload_hash) return io_fail(KVI_ERR_IO, p + ": payload hash mismatch");
    return KVI_OK;
}

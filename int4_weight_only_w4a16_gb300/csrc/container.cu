// The model container: this library's own on-disk format (layout in
// include/w4a16.h) -- a writer, a read-only memory-mapped reader that
// validates the header and directory, and an uploader that streams a tensor
// into device memory through two pinned staging buffers.
//
// "How to build your own LLM runtime from scratch (Towards Data Science)",
// "What it actually builds": packed INT4 weights in the engine's own
// memory-mapped binary file behind a magic-byte header.
#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <array>
#include <cerrno>
#include <cstring>
#include <string>
#include <vector>

#include "common.cuh"

namespace w4 {

constexpr char kMagic[8] = {'W', '4', 'A', '1', '6', 'M', 'C', '\0'};
constexpr uint32_t kVersion = 1;
constexpr size_t kPage = 4096;
constexpr size_t kEntryBytes = 112;
constexpr size_t kNameBytes = 64;
constexpr size_t kHeaderFixed = 8 + 4 + 4 + 8 + 7 * 4 + 2 * 4;   // before the header CRC
constexpr size_t kStageBytes = 8u << 20;
constexpr int kMaxTensors = 1 << 20;

// CRC-32, IEEE 802.3 (reflected polynomial 0xEDB88320).  Eight tables
// (slicing by 8): t[0] is the byte-at-a-time table, t[k][i] advances t[k-1][i]
// by one more zero byte, so eight input bytes fold in with eight lookups.
static const std::array<std::array<uint32_t, 256>, 8>& crc_tables() {
    static const std::array<std::array<uint32_t, 256>, 8> tables = [] {
        std::array<std::array<uint32_t, 256>, 8> t{};
        for (uint32_t i = 0; i < 256; ++i) {
            uint32_t c = i;
            for (int b = 0; b < 8; ++b) c = (c & 1u) ? (0xEDB88320u ^ (c >> 1)) : (c >> 1);
            t[0][i] = c;
        }
        for (int k = 1; k < 8; ++k)
            for (uint32_t i = 0; i < 256; ++i) t[k][i] = (t[k - 1][i] >> 8) ^ t[0][t[k - 1][i] & 0xFFu];
        return t;
    }();
    return tables;
}
static uint32_t crc32_update(uint32_t crc, const void* data, size_t n) {
    const auto& t = crc_tables();
    const unsigned char* p = static_cast<const unsigned char*>(data);
    while (n >= 8) {
        const uint32_t lo = crc ^ ((uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) |
                                   ((uint32_t)p[3] << 24));
        crc = t[7][lo & 0xFFu] ^ t[6][(lo >> 8) & 0xFFu] ^ t[5][(lo >> 16) & 0xFFu] ^ t[4][lo >> 24] ^
              t[3][p[4]] ^ t[2][p[5]] ^ t[1][p[6]] ^ t[0][p[7]];
        p += 8;
        n -= 8;
    }
    for (; n > 0; --n, ++p) crc = t[0][(crc ^ *p) & 0xFFu] ^ (crc >> 8);
    return crc;
}
static uint32_t crc32_of(const void* data, size_t n) { return crc32_update(0xFFFFFFFFu, data, n) ^ 0xFFFFFFFFu; }

// little-endian field access, byte by byte (no host-order assumptions)
static void put_u32(unsigned char* p, uint32_t v) {
    for (int i = 0; i < 4; ++i) p[i] = (unsigned char)(v >> (8 * i));
}
static void put_u64(unsigned char* p, uint64_t v) {
    for (int i = 0; i < 8; ++i) p[i] = (unsigned char)(v >> (8 * i));
}
static uint32_t get_u32(const unsigned char* p) {
    uint32_t v = 0;
    for (int i = 0; i < 4; ++i) v |= (uint32_t)p[i] << (8 * i);
    return v;
}
static uint64_t get_u64(const unsigned char* p) {
    uint64_t v = 0;
    for (int i = 0; i < 8; ++i) v |= (uint64_t)p[i] << (8 * i);
    return v;
}
static void put_f32(unsigned char* p, float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    put_u32(p, u);
}
static float get_f32(const unsigned char* p) {
    const uint32_t u = get_u32(p);
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}

static size_t dtype_bytes(int dt) {
    switch (dt) {
        case W4_DT_U32: return 4;
        case W4_DT_F16: return 2;
        case W4_DT_F32: return 4;
        case W4_DT_I32: return 4;
        default: return 0;
    }
}
static size_t align_page(size_t v) { return (v + kPage - 1) / kPage * kPage; }

struct Entry {
    std::string name;
    int dtype, ndim;
    int64_t dims[2];
    uint64_t offset, bytes;
    uint32_t crc;
};

static bool write_all(int fd, const void* data, size_t n) {
    const char* p = static_cast<const char*>(data);
    while (n > 0) {
        const ssize_t w = ::write(fd, p, n);
        if (w < 0) {
            if (errno == EINTR) continue;
            return false;
        }
        p += w;
        n -= (size_t)w;
    }
    return true;
}

}  // namespace w4

struct w4_container {
    int fd = -1;
    const unsigned char* map = nullptr;
    size_t map_bytes = 0;
    w4_model_config cfg = {};
    std::vector<w4::Entry> entries;
    void* stage[2] = {nullptr, nullptr};   // pinned staging buffers
    cudaEvent_t done[2] = {nullptr, nullptr};
    int device = -1;
};

extern "C" w4_status w4_container_write(const char* path, const w4_model_config* cfg, const w4_tensor_desc* tensors,
                                        int n_tensors) {
    using namespace w4;
    W4_REQUIRE(path && cfg && (tensors || n_tensors == 0), W4_ERR_NULL, "container_write: null pointer");
    W4_REQUIRE(n_tensors >= 0 && n_tensors <= kMaxTensors, W4_ERR_SHAPE, "container_write: %d tensors", n_tensors);
    std::vector<Entry> es((size_t)n_tensors);
    const size_t dir_end = kPage + (size_t)n_tensors * kEntryBytes;
    size_t off = align_page(dir_end);
    for (int i = 0; i < n_tensors; ++i) {
        const w4_tensor_desc& t = tensors[i];
        W4_REQUIRE(t.name && std::strlen(t.name) > 0 && std::strlen(t.name) < kNameBytes, W4_ERR_SHAPE,
                   "container_write: tensor %d needs a name of 1..%zu bytes", i, kNameBytes - 1);
        W4_REQUIRE(dtype_bytes(t.dtype) > 0, W4_ERR_SHAPE, "container_write: tensor '%s' has dtype %d", t.name,
                   t.dtype);
        W4_REQUIRE(t.ndim == 1 || t.ndim == 2, W4_ERR_SHAPE, "container_write: tensor '%s' has ndim %d", t.name,
                   t.ndim);
        const int64_t d1 = t.ndim == 2 ? t.dims[1] : 1;
        W4_REQUIRE(t.dims[0] > 0 && d1 > 0 && t.dims[0] < (1LL << 40) && d1 < (1LL << 40), W4_ERR_SHAPE,
                   "container_write: tensor '%s' has bad dims", t.name);
        const uint64_t nb = (uint64_t)t.dims[0] * (uint64_t)d1 * dtype_bytes(t.dtype);
        W4_REQUIRE(nb == t.bytes, W4_ERR_SHAPE, "container_write: tensor '%s' is %zu bytes, dims say %llu", t.name,
                   t.bytes, (unsigned long long)nb);
        W4_REQUIRE(t.data != nullptr, W4_ERR_NULL, "container_write: tensor '%s' has no data", t.name);
        for (int j = 0; j < i; ++j)
            W4_REQUIRE(es[j].name != t.name, W4_ERR_SHAPE, "container_write: duplicate tensor name '%s'", t.name);
        Entry& e = es[i];
        e.name = t.name;
        e.dtype = t.dtype;
        e.ndim = t.ndim;
        e.dims[0] = t.dims[0];
        e.dims[1] = t.ndim == 2 ? t.dims[1] : 0;
        e.offset = off;
        e.bytes = nb;
        e.crc = crc32_of(t.data, t.bytes);
        off = align_page(off + nb);
    }
    const uint64_t file_bytes = off;

    std::vector<unsigned char> head(align_page(dir_end), 0);
    unsigned char* h = head.data();
    std::memcpy(h, kMagic, 8);
    put_u32(h + 8, kVersion);
    put_u32(h + 12, (uint32_t)n_tensors);
    put_u64(h + 16, file_bytes);
    const int32_t ints[7] = {cfg->hidden, cfg->ffn, cfg->n_layers, cfg->n_q_heads, cfg->n_kv_heads, cfg->head_dim,
                             cfg->vocab};
    for (int i = 0; i < 7; ++i) put_u32(h + 24 + 4 * i, (uint32_t)ints[i]);
    put_f32(h + 52, cfg->rms_eps);
    put_f32(h + 56, cfg->rope_theta);
    put_u32(h + kHeaderFixed, crc32_of(h, kHeaderFixed));
    for (int i = 0; i < n_tensors; ++i) {
        unsigned char* e = h + kPage + (size_t)i * kEntryBytes;
        std::memcpy(e, es[i].name.c_str(), es[i].name.size());
        put_u32(e + 64, (uint32_t)es[i].dtype);
        put_u32(e + 68, (uint32_t)es[i].ndim);
        put_u64(e + 72, (uint64_t)es[i].dims[0]);
        put_u64(e + 80, (uint64_t)es[i].dims[1]);
        put_u64(e + 88, es[i].offset);
        put_u64(e + 96, es[i].bytes);
        put_u32(e + 104, es[i].crc);
    }

    const int fd = ::open(path, O_WRONLY | O_CREAT | O_TRUNC, 0644);
    W4_REQUIRE(fd >= 0, W4_ERR_IO, "container_write: cannot create '%s': %s", path, std::strerror(errno));
    bool ok = write_all(fd, head.data(), head.size());
    std::vector<unsigned char> zeros(kPage, 0);
    size_t pos = head.size();
    for (int i = 0; ok && i < n_tensors; ++i) {
        ok = write_all(fd, tensors[i].data, tensors[i].bytes);
        pos += tensors[i].bytes;
        const size_t pad = align_page(pos) - pos;
        if (ok && pad) ok = write_all(fd, zeros.data(), pad);
        pos += pad;
    }
    ok = ok && ::fsync(fd) == 0;
    ::close(fd);
    W4_REQUIRE(ok && pos == file_bytes, W4_ERR_IO, "container_write: writing '%s' failed: %s", path,
               std::strerror(errno));
    return W4_OK;
}

extern "C" void w4_container_close(w4_container* c) {
    if (!c) return;
    for (int i = 0; i < 2; ++i) {
        if (c->done[i]) {
            cudaEventSynchronize(c->done[i]);
            cudaEventDestroy(c->done[i]);
        }
        if (c->stage[i]) cudaFreeHost(c->stage[i]);
    }
    if (c->map) ::munmap(const_cast<unsigned char*>(c->map), c->map_bytes);
    if (c->fd >= 0) ::close(c->fd);
    delete c;
}

extern "C" w4_status w4_container_open(const char* path, int verify, w4_container** out) {
    using namespace w4;
    W4_REQUIRE(path && out, W4_ERR_NULL, "container_open: null pointer");
    *out = nullptr;
    w4_container* c = new w4_container();
    auto fail = [&](w4_status s) {
        w4_container_close(c);
        return s;
    };
    c->fd = ::open(path, O_RDONLY);
    if (c->fd < 0) return fail(set_error(W4_ERR_IO, "container_open: cannot open '%s': %s", path, std::strerror(errno)));
    struct stat st;
    if (::fstat(c->fd, &st) != 0 || st.st_size < (off_t)kPage)
        return fail(set_error(W4_ERR_IO, "container_open: '%s' is shorter than a header", path));
    c->map_bytes = (size_t)st.st_size;
    void* m = ::mmap(nullptr, c->map_bytes, PROT_READ, MAP_SHARED, c->fd, 0);
    if (m == MAP_FAILED) {
        c->map = nullptr;
        return fail(set_error(W4_ERR_IO, "container_open: mmap of '%s' failed: %s", path, std::strerror(errno)));
    }
    c->map = static_cast<const unsigned char*>(m);
    const unsigned char* h = c->map;
    if (std::memcmp(h, kMagic, 8) != 0) return fail(set_error(W4_ERR_IO, "container_open: bad magic in '%s'", path));
    if (get_u32(h + 8) != kVersion)
        return fail(set_error(W4_ERR_IO, "container_open: version %u, expected %u", get_u32(h + 8), kVersion));
    if (get_u32(h + kHeaderFixed) != crc32_of(h, kHeaderFixed))
        return fail(set_error(W4_ERR_IO, "container_open: header CRC mismatch in '%s'", path));
    const uint32_t n = get_u32(h + 12);
    const uint64_t file_bytes = get_u64(h + 16);
    if (file_bytes != c->map_bytes)
        return fail(set_error(W4_ERR_IO, "container_open: '%s' is %zu bytes, header says %llu", path, c->map_bytes,
                              (unsigned long long)file_bytes));
    if (n > (uint32_t)kMaxTensors || kPage + (uint64_t)n * kEntryBytes > file_bytes)
        return fail(set_error(W4_ERR_IO, "container_open: directory of %u entries does not fit", n));
    int32_t ints[7];
    for (int i = 0; i < 7; ++i) ints[i] = (int32_t)get_u32(h + 24 + 4 * i);
    c->cfg.hidden = ints[0];
    c->cfg.ffn = ints[1];
    c->cfg.n_layers = ints[2];
    c->cfg.n_q_heads = ints[3];
    c->cfg.n_kv_heads = ints[4];
    c->cfg.head_dim = ints[5];
    c->cfg.vocab = ints[6];
    c->cfg.rms_eps = get_f32(h + 52);
    c->cfg.rope_theta = get_f32(h + 56);
    const uint64_t data0 = align_page(kPage + (uint64_t)n * kEntryBytes);
    c->entries.resize(n);
    for (uint32_t i = 0; i < n; ++i) {
        const unsigned char* e = h + kPage + (size_t)i * kEntryBytes;
        if (std::memchr(e, 0, kNameBytes) == nullptr || e[0] == 0)
            return fail(set_error(W4_ERR_IO, "container_open: entry %u has no valid name", i));
        Entry& en = c->entries[i];
        en.name = reinterpret_cast<const char*>(e);
        en.dtype = (int)get_u32(e + 64);
        en.ndim = (int)get_u32(e + 68);
        en.dims[0] = (int64_t)get_u64(e + 72);
        en.dims[1] = (int64_t)get_u64(e + 80);
        en.offset = get_u64(e + 88);
        en.bytes = get_u64(e + 96);
        en.crc = get_u32(e + 104);
        const size_t eb = dtype_bytes(en.dtype);
        const bool shape_ok = eb > 0 && (en.ndim == 1 || en.ndim == 2) && en.dims[0] > 0 &&
                              en.dims[0] < (1LL << 40) &&
                              (en.ndim == 1 ? en.dims[1] == 0 : (en.dims[1] > 0 && en.dims[1] < (1LL << 40)));
        if (!shape_ok) return fail(set_error(W4_ERR_IO, "container_open: entry '%s' has a bad dtype/shape", en.name.c_str()));
        const uint64_t want = (uint64_t)en.dims[0] * (uint64_t)(en.ndim == 2 ? en.dims[1] : 1) * eb;
        if (want != en.bytes || en.offset % kPage != 0 || en.offset < data0 || en.offset > file_bytes ||
            en.bytes > file_bytes - en.offset)
            return fail(set_error(W4_ERR_IO, "container_open: entry '%s' lies outside the file or mis-sized",
                                  en.name.c_str()));
        for (uint32_t j = 0; j < i; ++j)
            if (c->entries[j].name == en.name)
                return fail(set_error(W4_ERR_IO, "container_open: duplicate entry '%s'", en.name.c_str()));
        if (verify && crc32_of(h + en.offset, en.bytes) != en.crc)
            return fail(set_error(W4_ERR_IO, "container_open: CRC mismatch in tensor '%s'", en.name.c_str()));
    }
    *out = c;
    return W4_OK;
}

extern "C" w4_status w4_container_config(const w4_container* c, w4_model_config* cfg) {
    W4_REQUIRE(c && cfg, W4_ERR_NULL, "container_config: null pointer");
    *cfg = c->cfg;
    return W4_OK;
}

extern "C" int w4_container_count(const w4_container* c) { return c ? (int)c->entries.size() : 0; }

extern "C" w4_status w4_container_tensor(const w4_container* c, int index, w4_tensor_desc* out) {
    W4_REQUIRE(c && out, W4_ERR_NULL, "container_tensor: null pointer");
    W4_REQUIRE(index >= 0 && index < (int)c->entries.size(), W4_ERR_RANGE, "container_tensor: index %d of %zu",
               index, c->entries.size());
    const w4::Entry& e = c->entries[index];
    out->name = e.name.c_str();
    out->dtype = e.dtype;
    out->ndim = e.ndim;
    out->dims[0] = e.dims[0];
    out->dims[1] = e.dims[1];
    out->data = c->map + e.offset;
    out->bytes = e.bytes;
    return W4_OK;
}

extern "C" w4_status w4_container_find(const w4_container* c, const char* name, int* index) {
    W4_REQUIRE(c && name && index, W4_ERR_NULL, "container_find: null pointer");
    for (size_t i = 0; i < c->entries.size(); ++i)
        if (c->entries[i].name == name) {
            *index = (int)i;
            return W4_OK;
        }
    return w4::set_error(W4_ERR_RANGE, "container_find: no tensor '%s'", name);
}

extern "C" w4_status w4_container_upload(w4_container* c, int index, void* dst, size_t dst_bytes, void* stream) {
    using namespace w4;
    W4_REQUIRE(c && dst, W4_ERR_NULL, "container_upload: null pointer");
    W4_REQUIRE(index >= 0 && index < (int)c->entries.size(), W4_ERR_RANGE, "container_upload: index %d of %zu",
               index, c->entries.size());
    const Entry& e = c->entries[index];
    W4_REQUIRE(dst_bytes >= e.bytes, W4_ERR_CAPACITY, "container_upload: '%s' needs %llu bytes, got %zu",
               e.name.c_str(), (unsigned long long)e.bytes, dst_bytes);
    int dev = -1;
    W4_CUDA(cudaGetDevice(&dev));
    if (c->stage[0] == nullptr || c->device != dev) {
        for (int i = 0; i < 2; ++i) {
            if (c->done[i]) {
                W4_CUDA(cudaEventSynchronize(c->done[i]));
                cudaEventDestroy(c->done[i]);
                c->done[i] = nullptr;
            }
            if (c->stage[i]) cudaFreeHost(c->stage[i]);
            c->stage[i] = nullptr;
        }
        for (int i = 0; i < 2; ++i) {
            W4_CUDA(cudaHostAlloc(&c->stage[i], kStageBytes, cudaHostAllocDefault));
            W4_CUDA(cudaEventCreateWithFlags(&c->done[i], cudaEventDisableTiming));
        }
        c->device = dev;
    }
    cudaStream_t st = (cudaStream_t)stream;
    const unsigned char* src = c->map + e.offset;
    unsigned char* d = static_cast<unsigned char*>(dst);
    int b = 0;
    for (uint64_t done = 0; done < e.bytes; b ^= 1) {
        const size_t n = (size_t)std::min<uint64_t>(kStageBytes, e.bytes - done);
        W4_CUDA(cudaEventSynchronize(c->done[b]));   // the copy that last used this buffer has finished
        std::memcpy(c->stage[b], src + done, n);
        W4_CUDA(cudaMemcpyAsync(d + done, c->stage[b], n, cudaMemcpyHostToDevice, st));
        W4_CUDA(cudaEventRecord(c->done[b], st));
        done += n;
    }
    return W4_OK;
}

// qk_gguf.cpp -- GGUF container reader (host code): the file the blocks come in.
//
// Layout ("12 -- llama.cpp / GGUF / Local Inference Mastery", "Part 1 -- The
// GGUF format (bit-level)", file structure figure): a header (magic "GGUF",
// version uint32, tensor_count uint64, metadata_kv_count uint64), the
// metadata key/value entries (length-prefixed key, value type, value), one
// info entry per tensor (name, n_dims, shape, type, offset), padding to the
// alignment (32 bytes unless the file says otherwise), then the tensor data at
// offsets from the start of that data section.  Little-endian throughout.
// The value-type codes, the ggml tensor-type numbers, the 64-bit string
// lengths of versions 2-3 and the "general.alignment" key are not on the page;
// they are the GGUF specification's, which the page cites.
//
// The reader parses an image in memory (a read-only mmap of the file, or a
// caller's buffer), checks every length, count and offset against the image
// before using it, and never copies tensor data: tensor info gives a pointer
// into the image.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <fcntl.h>
#include <string>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>
#include <vector>

#include "qk_internal.h"

namespace {

enum : uint32_t {   // metadata value types
    V_U8 = 0, V_I8 = 1, V_U16 = 2, V_I16 = 3, V_U32 = 4, V_I32 = 5, V_F32 = 6, V_BOOL = 7,
    V_STR = 8, V_ARR = 9, V_U64 = 10, V_I64 = 11, V_F64 = 12
};

enum : uint32_t {   // ggml tensor types this library sizes
    G_F32 = 0, G_F16 = 1, G_Q4_0 = 2, G_Q5_0 = 6, G_Q8_0 = 8, G_Q2_K = 10, G_Q3_K = 11, G_Q4_K = 12, G_Q5_K = 13, G_Q6_K = 14, G_BF16 = 30
};

constexpr int kMaxDims = 4;
constexpr int kMaxDepth = 8;   // nested arrays

// Bytes of a scalar value type (0: not a fixed-size scalar).
size_t scalar_size(uint32_t t) {
    switch (t) {
    case V_U8: case V_I8: case V_BOOL: return 1;
    case V_U16: case V_I16: return 2;
    case V_U32: case V_I32: case V_F32: return 4;
    case V_U64: case V_I64: case V_F64: return 8;
    }
    return 0;
}

// (block bytes, block elements, library type id or -1) of a ggml tensor type;
// block bytes 0 when this library does not know the type's size.
void ggml_block(uint32_t g, uint64_t& bb, uint64_t& be, int& qt) {
    qt = -1;
    switch (g) {
    case G_F32: bb = 4; be = 1; return;
    case G_F16: case G_BF16: bb = 2; be = 1; return;
    case G_Q4_0: bb = 18; be = 32; qt = QK_Q4_0; return;
    case G_Q5_0: bb = 22; be = 32; qt = QK_Q5_0; return;
    case G_Q8_0: bb = 34; be = 32; qt = QK_Q8_0; return;
    case G_Q4_K: bb = 144; be = 256; qt = QK_Q4_K; return;
    case G_Q5_K: bb = 176; be = 256; qt = QK_Q5_K; return;
    case G_Q2_K: bb = 84; be = 256; qt = QK_Q2_K; return;
    case G_Q3_K: bb = 110; be = 256; qt = QK_Q3_K; return;
    case G_Q6_K: bb = 210; be = 256; qt = QK_Q6_K; return;
    }
    bb = 0;
    be = 1;
}

struct Cursor {
    const uint8_t* p;
    uint64_t n, at;
    bool ok = true;
    const char* why = nullptr;   // set when the failure is not running out of bytes
    bool need(uint64_t k) {
        if (!ok || k > n - at) ok = false;
        return ok;
    }
    template <typename U> U rd() {
        U v{};
        if (need(sizeof(U))) {
            std::memcpy(&v, p + at, sizeof(U));   // little-endian host (x86-64, aarch64)
            at += sizeof(U);
        }
        return v;
    }
    bool skip(uint64_t k) {
        if (need(k)) at += k;
        return ok;
    }
};

struct KV {
    std::string key;
    uint32_t type = 0;
    uint64_t off = 0;                // value's offset in the image (after the type)
    uint32_t arr_type = 0;           // arrays: element type and count
    uint64_t arr_n = 0;
    uint64_t arr_off = 0;            // offset of the first element
    std::vector<uint64_t> str_offs;  // string arrays: offset of each element's length
};

struct Tensor {
    std::string name;
    uint32_t n_dims = 0;
    int64_t dims[kMaxDims] = {1, 1, 1, 1};
    uint32_t ggml_type = 0;
    int qk_type = -1;
    uint64_t offset = 0;   // from the start of the data section
    uint64_t nbytes = 0;   // 0 when the type's size is not known here
};

bool read_str(Cursor& c, std::string* out) {
    const uint64_t len = c.rd<uint64_t>();
    if (!c.need(len)) return false;
    if (out) out->assign(reinterpret_cast<const char*>(c.p + c.at), (size_t)len);
    c.at += len;
    return true;
}

// Skip one value of type t (arrays recursively, to kMaxDepth).
bool skip_value(Cursor& c, uint32_t t, int depth) {
    if (const size_t s = scalar_size(t)) return c.skip(s);
    if (t == V_STR) return read_str(c, nullptr);
    if (t != V_ARR) {
        c.why = "unknown metadata value type";
        return c.ok = false;
    }
    if (depth >= kMaxDepth) {
        c.why = "metadata arrays nested more than 8 deep";
        return c.ok = false;
    }
    const uint32_t et = c.rd<uint32_t>();
    const uint64_t n = c.rd<uint64_t>();
    if (!c.ok) return false;
    if (const size_t s = scalar_size(et)) return n <= (c.n - c.at) / s && c.skip(n * s);
    if (et != V_STR && et != V_ARR) {
        c.why = "unknown array element type";
        return c.ok = false;
    }
    if (n > (c.n - c.at) / 8) return c.ok = false;   // every element takes at least 8 bytes
    for (uint64_t i = 0; i < n; ++i)
        if (!skip_value(c, et, depth + 1)) return false;
    return true;
}

}  // namespace

struct qk_gguf {
    const uint8_t* image = nullptr;
    uint64_t size = 0;
    void* map = nullptr;   // non-null when the image is this handle's mmap
    uint32_t version = 0;
    uint64_t alignment = 32, data_off = 0;
    std::vector<KV> kv;
    std::vector<Tensor> tensors;
};

namespace {

qk_status parse(qk_gguf* g) {
    Cursor c{g->image, g->size, 0};
    if (g->size < 24 || std::memcmp(g->image, "GGUF", 4) != 0)
        return qk::set_error(QK_ERR_FORMAT, "not a GGUF image (magic)");
    c.at = 4;
    g->version = c.rd<uint32_t>();
    if (g->version < 2 || g->version > 3)
        return qk::set_error(QK_ERR_FORMAT, "unsupported GGUF version (2 and 3 are read)");
    const uint64_t nt = c.rd<uint64_t>(), nkv = c.rd<uint64_t>();
    // Each entry takes at least 12 (kv) or 24 (tensor) bytes: bound the counts
    // by the image before reserving anything.
    if (nkv > (g->size - c.at) / 12 || nt > (g->size - c.at) / 24)
        return qk::set_error(QK_ERR_FORMAT, "entry counts exceed the image");
    g->kv.resize((size_t)nkv);
    for (uint64_t i = 0; i < nkv; ++i) {
        KV& e = g->kv[(size_t)i];
        if (!read_str(c, &e.key)) break;
        e.type = c.rd<uint32_t>();
        e.off = c.at;
        if (!c.ok) break;
        if (e.type == V_ARR) {
            e.arr_type = c.rd<uint32_t>();
            e.arr_n = c.rd<uint64_t>();
            e.arr_off = c.at;
            if (!c.ok) break;
            if (e.arr_type == V_STR) {
                if (e.arr_n > (c.n - c.at) / 8) {
                    c.ok = false;
                    break;
                }
                e.str_offs.resize((size_t)e.arr_n);
                for (uint64_t j = 0; j < e.arr_n && c.ok; ++j) {
                    e.str_offs[(size_t)j] = c.at;
                    read_str(c, nullptr);
                }
            } else {
                c.at = e.off;
                skip_value(c, V_ARR, 0);
            }
        } else {
            skip_value(c, e.type, 0);
        }
        if (!c.ok) break;
        if (e.key == "general.alignment") {
            if (e.type != V_U32) return qk::set_error(QK_ERR_FORMAT, "general.alignment is not a uint32");
            uint32_t a = 0;
            std::memcpy(&a, g->image + e.off, 4);
            if (a == 0 || (a & (a - 1)) != 0 || a > (1u << 20))
                return qk::set_error(QK_ERR_FORMAT, "general.alignment is not a power of two <= 1 MiB");
            g->alignment = a;
        }
    }
    if (!c.ok) return qk::set_error(QK_ERR_FORMAT, c.why ? c.why : "metadata runs past the end of the image");
    g->tensors.resize((size_t)nt);
    for (uint64_t i = 0; i < nt; ++i) {
        Tensor& t = g->tensors[(size_t)i];
        if (!read_str(c, &t.name)) break;
        t.n_dims = c.rd<uint32_t>();
        if (!c.ok) break;
        if (t.n_dims < 1 || t.n_dims > kMaxDims)
            return qk::set_error(QK_ERR_FORMAT, "tensor n_dims outside 1..4");
        uint64_t ne = 1;
        for (uint32_t d = 0; d < t.n_dims; ++d) {
            const uint64_t v = c.rd<uint64_t>();
            if (v > (uint64_t)INT64_MAX || (v != 0 && ne > (uint64_t)INT64_MAX / v))
                return qk::set_error(QK_ERR_FORMAT, "tensor shape overflows");
            t.dims[d] = (int64_t)v;
            ne *= v;
        }
        t.ggml_type = c.rd<uint32_t>();
        t.offset = c.rd<uint64_t>();
        if (!c.ok) break;
        uint64_t bb, be;
        ggml_block(t.ggml_type, bb, be, t.qk_type);
        if (bb) {
            if ((uint64_t)t.dims[0] % be != 0)
                return qk::set_error(QK_ERR_FORMAT, "tensor rows are not whole blocks");
            if (ne / be > UINT64_MAX / bb) return qk::set_error(QK_ERR_FORMAT, "tensor size overflows");
            t.nbytes = ne / be * bb;
        }
        if (t.offset % g->alignment != 0) return qk::set_error(QK_ERR_FORMAT, "tensor offset is not aligned");
    }
    if (!c.ok) return qk::set_error(QK_ERR_FORMAT, "tensor infos run past the end of the image");
    // The data section starts at the next multiple of the alignment.
    const uint64_t a = g->alignment;
    g->data_off = (c.at + a - 1) / a * a;
    if (g->data_off > g->size && nt > 0) return qk::set_error(QK_ERR_FORMAT, "no room for the data section");
    for (const Tensor& t : g->tensors) {
        if (t.offset > g->size - std::min(g->size, g->data_off) || t.nbytes > g->size - g->data_off - t.offset)
            return qk::set_error(QK_ERR_FORMAT, "tensor data runs past the end of the image");
    }
    return QK_OK;
}

}  // namespace

extern "C" {

qk_status qk_gguf_parse(const void* data, uint64_t size, qk_gguf** out) {
    if (!out) return qk::set_error(QK_ERR_NULL, "out is NULL");
    *out = nullptr;
    if (!data) return qk::set_error(QK_ERR_NULL, "data is NULL");
    qk_gguf* g = new qk_gguf();
    g->image = static_cast<const uint8_t*>(data);
    g->size = size;
    const qk_status st = parse(g);
    if (st != QK_OK) {
        delete g;
        return st;
    }
    *out = g;
    return QK_OK;
}

qk_status qk_gguf_open(const char* path, qk_gguf** out) {
    if (!out) return qk::set_error(QK_ERR_NULL, "out is NULL");
    *out = nullptr;
    if (!path) return qk::set_error(QK_ERR_NULL, "path is NULL");
    const int fd = open(path, O_RDONLY);
    if (fd < 0) return qk::set_error(QK_ERR_IO, "cannot open the file");
    struct stat sb;
    if (fstat(fd, &sb) != 0 || sb.st_size <= 0) {
        close(fd);
        return qk::set_error(QK_ERR_IO, "cannot stat the file, or it is empty");
    }
    void* m = mmap(nullptr, (size_t)sb.st_size, PROT_READ, MAP_PRIVATE, fd, 0);
    close(fd);   // the mapping stays valid
    if (m == MAP_FAILED) return qk::set_error(QK_ERR_IO, "mmap failed");
    qk_gguf* g = nullptr;
    const qk_status st = qk_gguf_parse(m, (uint64_t)sb.st_size, &g);
    if (st != QK_OK) {
        munmap(m, (size_t)sb.st_size);
        return st;
    }
    g->map = m;
    *out = g;
    return QK_OK;
}

void qk_gguf_close(qk_gguf* g) {
    if (!g) return;
    if (g->map) munmap(g->map, (size_t)g->size);
    delete g;
}

uint32_t qk_gguf_version(const qk_gguf* g) { return g ? g->version : 0; }
int64_t qk_gguf_n_kv(const qk_gguf* g) { return g ? (int64_t)g->kv.size() : -1; }
int64_t qk_gguf_n_tensors(const qk_gguf* g) { return g ? (int64_t)g->tensors.size() : -1; }
uint64_t qk_gguf_alignment(const qk_gguf* g) { return g ? g->alignment : 0; }
uint64_t qk_gguf_data_offset(const qk_gguf* g) { return g ? g->data_off : 0; }
const void* qk_gguf_image(const qk_gguf* g) { return g ? g->image : nullptr; }

// ---------------------------------------------------------------- metadata --

static const KV* kv_at(const qk_gguf* g, int64_t i) {
    return (g && i >= 0 && i < (int64_t)g->kv.size()) ? &g->kv[(size_t)i] : nullptr;
}

int64_t qk_gguf_find_kv(const qk_gguf* g, const char* key) {
    if (!g || !key) return -1;
    for (size_t i = 0; i < g->kv.size(); ++i)
        if (g->kv[i].key == key) return (int64_t)i;
    return -1;
}

const char* qk_gguf_kv_key(const qk_gguf* g, int64_t i) {
    const KV* e = kv_at(g, i);
    return e ? e->key.c_str() : nullptr;
}

int qk_gguf_kv_type(const qk_gguf* g, int64_t i) {
    const KV* e = kv_at(g, i);
    return e ? (int)e->type : -1;
}

// Integer (any width, signed or not) or bool value of scalar type t at p.
static bool scalar_int(const uint8_t* p, uint32_t t, int64_t* v) {
    switch (t) {
    case V_U8: case V_BOOL: *v = p[0]; return true;
    case V_I8: *v = (int8_t)p[0]; return true;
    case V_U16: { uint16_t x; std::memcpy(&x, p, 2); *v = x; return true; }
    case V_I16: { int16_t x; std::memcpy(&x, p, 2); *v = x; return true; }
    case V_U32: { uint32_t x; std::memcpy(&x, p, 4); *v = x; return true; }
    case V_I32: { int32_t x; std::memcpy(&x, p, 4); *v = x; return true; }
    case V_I64: { int64_t x; std::memcpy(&x, p, 8); *v = x; return true; }
    case V_U64: {
        uint64_t x;
        std::memcpy(&x, p, 8);
        if (x > (uint64_t)INT64_MAX) return false;
        *v = (int64_t)x;
        return true;
    }
    }
    return false;
}

static bool scalar_float(const uint8_t* p, uint32_t t, double* v) {
    if (t == V_F32) { float x; std::memcpy(&x, p, 4); *v = x; return true; }
    if (t == V_F64) { std::memcpy(v, p, 8); return true; }
    return false;
}

qk_status qk_gguf_kv_int(const qk_gguf* g, int64_t i, int64_t* v) {
    const KV* e = kv_at(g, i);
    if (!e || !v) return qk::set_error(QK_ERR_ARG, "no such key, or v is NULL");
    if (!scalar_int(g->image + e->off, e->type, v))
        return qk::set_error(QK_ERR_TYPE, "value is not an integer or bool (or a uint64 beyond int64)");
    return QK_OK;
}

qk_status qk_gguf_kv_float(const qk_gguf* g, int64_t i, double* v) {
    const KV* e = kv_at(g, i);
    if (!e || !v) return qk::set_error(QK_ERR_ARG, "no such key, or v is NULL");
    if (!scalar_float(g->image + e->off, e->type, v)) return qk::set_error(QK_ERR_TYPE, "value is not a float");
    return QK_OK;
}

static const char* str_at(const qk_gguf* g, uint64_t off, uint64_t* len) {
    uint64_t n;
    std::memcpy(&n, g->image + off, 8);   // checked while parsing
    if (len) *len = n;
    return reinterpret_cast<const char*>(g->image + off + 8);
}

const char* qk_gguf_kv_str(const qk_gguf* g, int64_t i, uint64_t* len) {
    const KV* e = kv_at(g, i);
    if (!e || e->type != V_STR) return nullptr;
    return str_at(g, e->off, len);
}

qk_status qk_gguf_kv_array(const qk_gguf* g, int64_t i, int* elem_type, uint64_t* n) {
    const KV* e = kv_at(g, i);
    if (!e) return qk::set_error(QK_ERR_ARG, "no such key");
    if (e->type != V_ARR) return qk::set_error(QK_ERR_TYPE, "value is not an array");
    if (elem_type) *elem_type = (int)e->arr_type;
    if (n) *n = e->arr_n;
    return QK_OK;
}

qk_status qk_gguf_kv_array_int(const qk_gguf* g, int64_t i, uint64_t j, int64_t* v) {
    const KV* e = kv_at(g, i);
    if (!e || e->type != V_ARR || j >= e->arr_n || !v) return qk::set_error(QK_ERR_ARG, "no such array element");
    const size_t s = scalar_size(e->arr_type);
    if (!s || !scalar_int(g->image + e->arr_off + j * s, e->arr_type, v))
        return qk::set_error(QK_ERR_TYPE, "element is not an integer or bool");
    return QK_OK;
}

qk_status qk_gguf_kv_array_float(const qk_gguf* g, int64_t i, uint64_t j, double* v) {
    const KV* e = kv_at(g, i);
    if (!e || e->type != V_ARR || j >= e->arr_n || !v) return qk::set_error(QK_ERR_ARG, "no such array element");
    const size_t s = scalar_size(e->arr_type);
    if (!s || !scalar_float(g->image + e->arr_off + j * s, e->arr_type, v))
        return qk::set_error(QK_ERR_TYPE, "element is not a float");
    return QK_OK;
}

const char* qk_gguf_kv_array_str(const qk_gguf* g, int64_t i, uint64_t j, uint64_t* len) {
    const KV* e = kv_at(g, i);
    if (!e || e->type != V_ARR || e->arr_type != V_STR || j >= e->arr_n) return nullptr;
    return str_at(g, e->str_offs[(size_t)j], len);
}

// ----------------------------------------------------------------- tensors --

int64_t qk_gguf_find_tensor(const qk_gguf* g, const char* name) {
    if (!g || !name) return -1;
    for (size_t i = 0; i < g->tensors.size(); ++i)
        if (g->tensors[i].name == name) return (int64_t)i;
    return -1;
}

qk_status qk_gguf_tensor(const qk_gguf* g, int64_t i, qk_gguf_tensor_info* info) {
    if (!g || !info || i < 0 || i >= (int64_t)g->tensors.size())
        return qk::set_error(QK_ERR_ARG, "no such tensor, or info is NULL");
    const Tensor& t = g->tensors[(size_t)i];
    info->name = t.name.c_str();
    info->n_dims = t.n_dims;
    for (int d = 0; d < kMaxDims; ++d) info->dims[d] = t.dims[d];
    info->ggml_type = t.ggml_type;
    info->qk_type = t.qk_type;
    info->offset = g->data_off + t.offset;
    info->nbytes = t.nbytes;
    info->data = g->image + g->data_off + t.offset;
    return QK_OK;
}

}  // extern "C"

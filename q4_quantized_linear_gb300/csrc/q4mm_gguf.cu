// q4mm_gguf.cu -- a reader of GGUF files in front of q4_0_pack (host code).
//
// "Go AI Inference: What is Inference?", section "GGUF: The Whole Model in
// One File": a GGUF file opens with the magic bytes GGUF, a version and two
// counts (tensors, metadata entries); then come the metadata (typed
// key-value pairs: scalars, strings and homogeneous arrays), the tensor
// descriptors (name, shape, type and an offset, no data) and the data blob
// the offsets point into. Section "The blob: getting the weights into
// memory": a loader parses only the header, the metadata and the
// descriptors first, then places each tensor's bytes where it goes -- here,
// the caller reads one tensor's bytes into host memory, copies them to the
// device and packs them with q4_0_pack.
//
// The page draws the layout but does not list the field widths and type
// codes; those follow GGUF version 2 and 3 as ggml writes them (the page
// points at ggml's gguf.h): little-endian, u32 version, u64 counts, strings
// as u64 length + bytes, value types 0..12 (u8, i8, u16, i16, u32, i32, f32,
// bool, string, array, u64, i64, f64), a tensor descriptor as name, u32 dim
// count, u64 dims (innermost first), u32 tensor type, u64 offset; the data
// blob starts at the first multiple of general.alignment (default 32) after
// the descriptors. Every size read from the file is checked against the
// file before it is used; a file that breaks a rule is refused with
// Q4_ERR_FORMAT, and nothing is read past its end.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/q4mm.h"

namespace {

constexpr uint32_t kTypeU8 = 0, kTypeI8 = 1, kTypeU16 = 2, kTypeI16 = 3, kTypeU32 = 4, kTypeI32 = 5,
                   kTypeF32 = 6, kTypeBool = 7, kTypeString = 8, kTypeArray = 9, kTypeU64 = 10,
                   kTypeI64 = 11, kTypeF64 = 12;
constexpr int kMaxDims = 4;

struct Tensor {
    std::string name;
    int type = 0;
    int n_dims = 0;
    int64_t dims[kMaxDims] = {1, 1, 1, 1};
    uint64_t offset = 0;   // from the start of the data blob
    uint64_t bytes = 0;    // 0 when the type's size is not known here
};

struct KV {
    std::string key;
    uint32_t type = 0;
    int64_t ivalue = 0;    // integer and bool scalars
    std::string svalue;    // strings
};

// Bytes of n elements of a tensor type, for the types whose size is fixed
// here (0 for the others): f32, f16, Q4_0 (18 bytes per 32), Q8_0 (34 per 32).
uint64_t tensor_bytes(int type, uint64_t n)
{
    switch (type) {
    case 0: return n * 4;
    case 1: return n * 2;
    case 2: return n % 32 ? 0 : n / 32 * 18;
    case 8: return n % 32 ? 0 : n / 32 * 34;
    default: return 0;
    }
}

// Sequential reader of the file's header; every read is bounds-checked.
class Reader {
public:
    Reader(FILE *f, uint64_t size) : f_(f), size_(size) {}
    bool bytes(void *dst, uint64_t n)
    {
        if (n > size_ - pos_) return false;
        if (n && fread(dst, 1, n, f_) != n) return false;
        pos_ += n;
        return true;
    }
    template <typename T> bool get(T *v)
    {
        uint8_t b[sizeof(T)];
        if (!bytes(b, sizeof(T))) return false;
        uint64_t u = 0;
        for (size_t i = 0; i < sizeof(T); ++i) u |= static_cast<uint64_t>(b[i]) << (8 * i);   // little endian
        std::memcpy(v, &u, sizeof(T));
        return true;
    }
    bool str(std::string *s)
    {
        uint64_t len = 0;
        if (!get(&len) || len > size_ - pos_) return false;
        s->resize(len);
        return bytes(len ? &(*s)[0] : nullptr, len);
    }
    bool skip(uint64_t n)
    {
        if (n > size_ - pos_) return false;
        if (n && fseek(f_, static_cast<long>(pos_ + n), SEEK_SET) != 0) return false;
        pos_ += n;
        return true;
    }
    uint64_t pos() const { return pos_; }
    uint64_t size() const { return size_; }

private:
    FILE *f_;
    uint64_t size_;
    uint64_t pos_ = 0;
};

uint64_t scalar_size(uint32_t type)
{
    switch (type) {
    case kTypeU8: case kTypeI8: case kTypeBool: return 1;
    case kTypeU16: case kTypeI16: return 2;
    case kTypeU32: case kTypeI32: case kTypeF32: return 4;
    case kTypeU64: case kTypeI64: case kTypeF64: return 8;
    default: return 0;
    }
}

bool read_int(Reader &r, uint32_t type, int64_t *v)
{
    switch (type) {
    case kTypeU8: { uint8_t x; if (!r.get(&x)) return false; *v = x; return true; }
    case kTypeI8: { int8_t x; if (!r.get(&x)) return false; *v = x; return true; }
    case kTypeBool: { uint8_t x; if (!r.get(&x) || x > 1) return false; *v = x; return true; }
    case kTypeU16: { uint16_t x; if (!r.get(&x)) return false; *v = x; return true; }
    case kTypeI16: { int16_t x; if (!r.get(&x)) return false; *v = x; return true; }
    case kTypeU32: { uint32_t x; if (!r.get(&x)) return false; *v = x; return true; }
    case kTypeI32: { int32_t x; if (!r.get(&x)) return false; *v = x; return true; }
    case kTypeU64: { uint64_t x; if (!r.get(&x) || x > static_cast<uint64_t>(INT64_MAX)) return false; *v = static_cast<int64_t>(x); return true; }
    case kTypeI64: { int64_t x; if (!r.get(&x)) return false; *v = x; return true; }
    default: return false;
    }
}

} // namespace

struct q4_gguf {
    std::string path;
    uint32_t version = 0;
    uint64_t alignment = 32;
    uint64_t data_start = 0;
    uint64_t file_size = 0;
    std::vector<KV> kvs;
    std::vector<Tensor> tensors;
};

namespace {

int parse(FILE *f, uint64_t size, q4_gguf *g)
{
    Reader r(f, size);
    char magic[4];
    if (!r.bytes(magic, 4) || std::memcmp(magic, "GGUF", 4) != 0) return Q4_ERR_FORMAT;
    uint64_t n_tensors = 0, n_kv = 0;
    if (!r.get(&g->version) || (g->version != 2 && g->version != 3)) return Q4_ERR_FORMAT;
    if (!r.get(&n_tensors) || !r.get(&n_kv)) return Q4_ERR_FORMAT;
    // every entry takes at least 8 bytes of the file
    if (n_kv > size / 8 || n_tensors > size / 8) return Q4_ERR_FORMAT;
    for (uint64_t i = 0; i < n_kv; ++i) {
        KV kv;
        if (!r.str(&kv.key) || !r.get(&kv.type)) return Q4_ERR_FORMAT;
        if (kv.type == kTypeString) {
            if (!r.str(&kv.svalue)) return Q4_ERR_FORMAT;
        } else if (kv.type == kTypeArray) {
            uint32_t et = 0;
            uint64_t count = 0;
            if (!r.get(&et) || !r.get(&count)) return Q4_ERR_FORMAT;
            if (et == kTypeString) {
                for (uint64_t e = 0; e < count; ++e) {
                    uint64_t len = 0;
                    if (!r.get(&len) || !r.skip(len)) return Q4_ERR_FORMAT;
                }
            } else {
                const uint64_t es = scalar_size(et);
                if (es == 0 || count > (r.size() - r.pos()) / es || !r.skip(count * es)) return Q4_ERR_FORMAT;
            }
        } else if (kv.type == kTypeF32 || kv.type == kTypeF64) {
            if (!r.skip(scalar_size(kv.type))) return Q4_ERR_FORMAT;
        } else if (!read_int(r, kv.type, &kv.ivalue)) {
            return Q4_ERR_FORMAT;
        }
        if (kv.key == "general.alignment") {
            if (kv.type != kTypeU32 || kv.ivalue <= 0 || (kv.ivalue & (kv.ivalue - 1)) != 0) return Q4_ERR_FORMAT;
            g->alignment = static_cast<uint64_t>(kv.ivalue);
        }
        g->kvs.push_back(std::move(kv));
    }
    for (uint64_t i = 0; i < n_tensors; ++i) {
        Tensor t;
        uint32_t nd = 0, type = 0;
        if (!r.str(&t.name) || !r.get(&nd) || nd < 1 || nd > kMaxDims) return Q4_ERR_FORMAT;
        t.n_dims = static_cast<int>(nd);
        uint64_t elems = 1;
        for (uint32_t d = 0; d < nd; ++d) {
            uint64_t v = 0;
            if (!r.get(&v) || v == 0 || v > (uint64_t(1) << 40) || elems > (uint64_t(1) << 50) / v) return Q4_ERR_FORMAT;
            t.dims[d] = static_cast<int64_t>(v);
            elems *= v;
        }
        if (!r.get(&type) || type > 1024 || !r.get(&t.offset)) return Q4_ERR_FORMAT;
        t.type = static_cast<int>(type);
        if (t.offset % g->alignment != 0) return Q4_ERR_FORMAT;
        t.bytes = tensor_bytes(t.type, elems);
        g->tensors.push_back(std::move(t));
    }
    g->data_start = (r.pos() + g->alignment - 1) / g->alignment * g->alignment;
    g->file_size = size;
    for (const Tensor &t : g->tensors) {
        if (t.offset > size || g->data_start > size - t.offset || t.bytes > size - g->data_start - t.offset)
            return Q4_ERR_FORMAT;   // descriptor points past the end of the file
    }
    return Q4_OK;
}

const KV *find_kv(const q4_gguf *g, const char *key)
{
    for (const KV &kv : g->kvs)
        if (kv.key == key) return &kv;
    return nullptr;
}

} // namespace

extern "C" {

Q4MM_API int q4_gguf_open(const char *path, q4_gguf **out)
{
    if (!path || !out) return Q4_ERR_INVALID_ARG;
    *out = nullptr;
    FILE *f = fopen(path, "rb");
    if (!f) return Q4_ERR_IO;
    int rc = Q4_ERR_IO;
    if (fseek(f, 0, SEEK_END) == 0) {
        const long end = ftell(f);
        if (end >= 0 && fseek(f, 0, SEEK_SET) == 0) {
            q4_gguf *g = new (std::nothrow) q4_gguf;
            if (!g) {
                rc = Q4_ERR_NO_MEMORY;
            } else {
                g->path = path;
                rc = parse(f, static_cast<uint64_t>(end), g);
                if (rc == Q4_OK) *out = g;
                else delete g;
            }
        }
    }
    fclose(f);
    return rc;
}

Q4MM_API void q4_gguf_close(q4_gguf *g) { delete g; }

Q4MM_API int64_t q4_gguf_tensor_count(const q4_gguf *g) { return g ? static_cast<int64_t>(g->tensors.size()) : -1; }

Q4MM_API int64_t q4_gguf_find_tensor(const q4_gguf *g, const char *name)
{
    if (!g || !name) return -1;
    for (size_t i = 0; i < g->tensors.size(); ++i)
        if (g->tensors[i].name == name) return static_cast<int64_t>(i);
    return -1;
}

Q4MM_API int q4_gguf_tensor_info(const q4_gguf *g, int64_t index, const char **name, int *type, int *n_dims,
                                 int64_t *dims, uint64_t *file_offset, uint64_t *bytes)
{
    if (!g || index < 0 || index >= static_cast<int64_t>(g->tensors.size())) return Q4_ERR_INVALID_ARG;
    const Tensor &t = g->tensors[static_cast<size_t>(index)];
    if (name) *name = t.name.c_str();
    if (type) *type = t.type;
    if (n_dims) *n_dims = t.n_dims;
    if (dims)
        for (int d = 0; d < kMaxDims; ++d) dims[d] = t.dims[d];
    if (file_offset) *file_offset = g->data_start + t.offset;
    if (bytes) *bytes = t.bytes;
    return Q4_OK;
}

Q4MM_API int q4_gguf_read_tensor(const q4_gguf *g, int64_t index, void *host_dst, uint64_t dst_bytes)
{
    if (!g || !host_dst || index < 0 || index >= static_cast<int64_t>(g->tensors.size())) return Q4_ERR_INVALID_ARG;
    const Tensor &t = g->tensors[static_cast<size_t>(index)];
    if (t.bytes == 0 || dst_bytes < t.bytes) return Q4_ERR_INVALID_ARG;
    FILE *f = fopen(g->path.c_str(), "rb");
    if (!f) return Q4_ERR_IO;
    int rc = Q4_OK;
    const uint64_t at = g->data_start + t.offset;
    if (at > static_cast<uint64_t>(INT64_MAX) || fseek(f, static_cast<long>(at), SEEK_SET) != 0 ||
        fread(host_dst, 1, t.bytes, f) != t.bytes)
        rc = Q4_ERR_IO;   // the file changed since it was opened
    fclose(f);
    return rc;
}

Q4MM_API int q4_gguf_get_int(const q4_gguf *g, const char *key, int64_t *value)
{
    if (!g || !key || !value) return Q4_ERR_INVALID_ARG;
    const KV *kv = find_kv(g, key);
    if (!kv || scalar_size(kv->type) == 0 || kv->type == kTypeF32 || kv->type == kTypeF64) return Q4_ERR_INVALID_ARG;
    *value = kv->ivalue;
    return Q4_OK;
}

Q4MM_API int q4_gguf_get_string(const q4_gguf *g, const char *key, const char **value)
{
    if (!g || !key || !value) return Q4_ERR_INVALID_ARG;
    const KV *kv = find_kv(g, key);
    if (!kv || kv->type != kTypeString) return Q4_ERR_INVALID_ARG;
    *value = kv->svalue.c_str();
    return Q4_OK;
}

} // extern "C"

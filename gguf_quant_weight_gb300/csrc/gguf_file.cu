// GGUF container reader (host code): the metadata key-value pairs and the
// tensor table of a .gguf file, and each tensor's bytes, so that a weight
// stored in the file can be handed to the matmul entry points as it is.
//
// GGUF Support Proposal for mobius, 1.1 "Overview" (a single file holding the
// model metadata as key-value pairs and the tensor data with a per-tensor
// quantization type) and 3.2 / 3.3 (a reader lists the tensors with their
// names, types and data).  The binary layout read here is the published GGUF
// container format (version 2 and 3), little-endian:
//   u32 magic "GGUF", u32 version, u64 tensor count, u64 key-value count,
//   key-value pairs  {string key, u32 value type, value},
//   tensor infos     {string name, u32 n_dims, u64 dims[n_dims], u32 type, u64 offset},
//   padding to the alignment (key general.alignment, default 32),
//   tensor data: tensor i at data start + offset_i.
// A string is {u64 length, bytes}; an array is {u32 element type, u64 count,
// elements}.  dims[0] is the innermost (contiguous) dimension: a weight
// W[N, K] is stored with dims {K, N}.
//
// Every read is checked against the file's size; a malformed file gives
// GGUF_ERR_FORMAT, never an out-of-bounds access.
#include <cstdint>
#include <cstring>
#include <string>
#include <vector>
#include <new>

#include <fcntl.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include "../../include/gguf_mm.h"

namespace {

enum ValueType : uint32_t {
    VT_U8 = 0, VT_I8 = 1, VT_U16 = 2, VT_I16 = 3, VT_U32 = 4, VT_I32 = 5, VT_F32 = 6, VT_BOOL = 7,
    VT_STRING = 8, VT_ARRAY = 9, VT_U64 = 10, VT_I64 = 11, VT_F64 = 12
};

int scalar_size(uint32_t t) {
    switch (t) {
        case VT_U8: case VT_I8: case VT_BOOL: return 1;
        case VT_U16: case VT_I16: return 2;
        case VT_U32: case VT_I32: case VT_F32: return 4;
        case VT_U64: case VT_I64: case VT_F64: return 8;
        default: return 0;
    }
}

// Block values and bytes of the tensor types whose byte size is known here
// (F32, F16, BF16 and the block formats); 0 for the others.
void type_geometry(uint32_t t, int64_t* bv, int64_t* bb) {
    switch (t) {
        case 0: *bv = 1; *bb = 4; return;     // F32
        case 1: *bv = 1; *bb = 2; return;     // F16
        case 30: *bv = 1; *bb = 2; return;    // BF16
        case 2: *bv = 32; *bb = 18; return;   // Q4_0
        case 3: *bv = 32; *bb = 20; return;   // Q4_1
        case 6: *bv = 32; *bb = 22; return;   // Q5_0
        case 7: *bv = 32; *bb = 24; return;   // Q5_1
        case 8: *bv = 32; *bb = 34; return;   // Q8_0
        case 10: *bv = 256; *bb = 84; return;   // Q2_K
        case 11: *bv = 256; *bb = 110; return;  // Q3_K
        case 12: *bv = 256; *bb = 144; return;  // Q4_K
        case 13: *bv = 256; *bb = 176; return;  // Q5_K
        case 14: *bv = 256; *bb = 210; return;  // Q6_K
        default: *bv = 0; *bb = 0; return;
    }
}

struct Value {
    uint32_t type = 0;
    uint64_t pos = 0;      // file offset of the value (for arrays: of the first element)
    uint32_t elem = 0;     // arrays: element type
    uint64_t count = 0;    // arrays: element count; strings: byte length
};

struct KV {
    std::string key;
    Value v;
};

struct Tensor {
    std::string name;
    uint32_t type = 0;
    uint32_t n_dims = 0;
    int64_t dims[4] = {1, 1, 1, 1};
    uint64_t offset = 0;   // absolute file offset of the data
    uint64_t nbytes = 0;   // 0 when the type's size is unknown here
};

struct Cursor {
    const uint8_t* base;
    uint64_t size, pos;
    bool ok;
    bool need(uint64_t n) {
        if (!ok || n > size || pos > size - n) ok = false;
        return ok;
    }
    template <class T>
    T get() {
        T v{};
        if (need(sizeof(T))) {
            std::memcpy(&v, base + pos, sizeof(T));
            pos += sizeof(T);
        }
        return v;
    }
    bool skip(uint64_t n) {
        if (need(n)) pos += n;
        return ok;
    }
    bool str(std::string* out) {
        const uint64_t n = get<uint64_t>();
        if (!need(n)) return false;
        if (out) out->assign(reinterpret_cast<const char*>(base + pos), n);
        pos += n;
        return true;
    }
};

}  // namespace

struct gguf_file {
    int fd = -1;
    const uint8_t* map = nullptr;
    uint64_t size = 0;
    uint32_t version = 0;
    uint64_t alignment = 32;
    uint64_t data_start = 0;
    std::vector<KV> kv;
    std::vector<Tensor> tensors;
};

namespace {

// A value at the cursor: records where it is and skips over it.
bool read_value(Cursor& c, uint32_t type, Value* v, int depth) {
    v->type = type;
    if (type == VT_STRING) {
        const uint64_t n = c.get<uint64_t>();
        v->count = n;
        v->pos = c.pos;
        return c.skip(n);
    }
    if (type == VT_ARRAY) {
        if (depth > 0) return false;   // arrays of arrays: not used by the format's writers
        v->elem = c.get<uint32_t>();
        v->count = c.get<uint64_t>();
        v->pos = c.pos;
        if (!c.ok) return false;
        if (v->elem == VT_STRING) {
            for (uint64_t i = 0; i < v->count; ++i)
                if (!c.str(nullptr)) return false;
            return true;
        }
        const int es = scalar_size(v->elem);
        if (es == 0 || v->count > c.size / (uint64_t)es) return false;
        return c.skip(v->count * (uint64_t)es);
    }
    const int sz = scalar_size(type);
    if (sz == 0) return false;
    v->pos = c.pos;
    return c.skip((uint64_t)sz);
}

int parse(gguf_file* f) {
    Cursor c{f->map, f->size, 0, true};
    const uint32_t magic = c.get<uint32_t>();
    if (!c.ok || magic != 0x46554747u) return GGUF_ERR_FORMAT;   // bytes 'G' 'G' 'U' 'F'
    f->version = c.get<uint32_t>();
    if (f->version != 2 && f->version != 3) return GGUF_ERR_FORMAT;
    const uint64_t n_tensors = c.get<uint64_t>(), n_kv = c.get<uint64_t>();
    if (!c.ok || n_tensors > f->size / 24 || n_kv > f->size / 12) return GGUF_ERR_FORMAT;
    f->kv.reserve(n_kv);
    for (uint64_t i = 0; i < n_kv; ++i) {
        KV e;
        if (!c.str(&e.key)) return GGUF_ERR_FORMAT;
        const uint32_t t = c.get<uint32_t>();
        if (!c.ok || !read_value(c, t, &e.v, 0)) return GGUF_ERR_FORMAT;
        if (e.key == "general.alignment") {
            uint64_t a = 0;
            if (t == VT_U32) { uint32_t v; std::memcpy(&v, f->map + e.v.pos, 4); a = v; }
            else if (t == VT_U64) std::memcpy(&a, f->map + e.v.pos, 8);
            else return GGUF_ERR_FORMAT;
            if (a == 0 || (a & (a - 1)) != 0 || a > (1u << 20)) return GGUF_ERR_FORMAT;
            f->alignment = a;
        }
        f->kv.push_back(std::move(e));
    }
    f->tensors.reserve(n_tensors);
    for (uint64_t i = 0; i < n_tensors; ++i) {
        Tensor t;
        if (!c.str(&t.name)) return GGUF_ERR_FORMAT;
        t.n_dims = c.get<uint32_t>();
        if (!c.ok || t.n_dims < 1 || t.n_dims > 4) return GGUF_ERR_FORMAT;
        for (uint32_t d = 0; d < t.n_dims; ++d) {
            const uint64_t v = c.get<uint64_t>();
            if (v == 0 || v > (uint64_t(1) << 40)) return GGUF_ERR_FORMAT;
            t.dims[d] = (int64_t)v;
        }
        t.type = c.get<uint32_t>();
        t.offset = c.get<uint64_t>();
        if (!c.ok) return GGUF_ERR_FORMAT;
        f->tensors.push_back(std::move(t));
    }
    // tensor data: after the header, padded to the alignment
    f->data_start = (c.pos + f->alignment - 1) / f->alignment * f->alignment;
    for (Tensor& t : f->tensors) {
        if (t.offset % f->alignment != 0) return GGUF_ERR_FORMAT;
        int64_t bv, bb;
        type_geometry(t.type, &bv, &bb);
        if (bv > 0) {
            if (t.dims[0] % bv != 0) return GGUF_ERR_FORMAT;
            // bytes = dims[0]/bv * bb * dims[1] * dims[2] * dims[3], each step checked against 2^62
            uint64_t n = (uint64_t)(t.dims[0] / bv) * (uint64_t)bb;
            for (uint32_t d = 1; d < 4; ++d) {
                if (n > (uint64_t(1) << 62) / (uint64_t)t.dims[d]) return GGUF_ERR_FORMAT;
                n *= (uint64_t)t.dims[d];
            }
            t.nbytes = n;
        }
        if (t.offset > f->size || f->data_start > f->size - t.offset) return GGUF_ERR_FORMAT;
        t.offset += f->data_start;
        if (t.nbytes > f->size - t.offset) return GGUF_ERR_FORMAT;   // data past the end of the file
    }
    return GGUF_OK;
}

const KV* find_kv(const gguf_file* f, const char* key) {
    for (const KV& e : f->kv)
        if (e.key == key) return &e;
    return nullptr;
}

}  // namespace

extern "C" {

int gguf_file_open(const char* path, gguf_file_t* out) {
    if (!path || !out) return GGUF_ERR_INVALID_ARG;
    *out = nullptr;
    const int fd = open(path, O_RDONLY);
    if (fd < 0) return GGUF_ERR_IO;
    struct stat st;
    if (fstat(fd, &st) != 0) {
        close(fd);
        return GGUF_ERR_IO;
    }
    if (st.st_size <= 0) {   // empty (or not a regular file): no header to read
        close(fd);
        return GGUF_ERR_FORMAT;
    }
    void* m = mmap(nullptr, (size_t)st.st_size, PROT_READ, MAP_PRIVATE, fd, 0);
    if (m == MAP_FAILED) {
        close(fd);
        return GGUF_ERR_IO;
    }
    gguf_file* f = new (std::nothrow) gguf_file;
    if (!f) {
        munmap(m, (size_t)st.st_size);
        close(fd);
        return GGUF_ERR_IO;
    }
    f->fd = fd;
    f->map = static_cast<const uint8_t*>(m);
    f->size = (uint64_t)st.st_size;
    const int rc = parse(f);
    if (rc != GGUF_OK) {
        gguf_file_close(f);
        return rc;
    }
    *out = f;
    return GGUF_OK;
}

void gguf_file_close(gguf_file_t f) {
    if (!f) return;
    if (f->map) munmap(const_cast<uint8_t*>(f->map), (size_t)f->size);
    if (f->fd >= 0) close(f->fd);
    delete f;
}

int gguf_file_version(gguf_file_t f) { return f ? (int)f->version : GGUF_ERR_INVALID_ARG; }

int64_t gguf_file_alignment(gguf_file_t f) { return f ? (int64_t)f->alignment : GGUF_ERR_INVALID_ARG; }

int64_t gguf_file_tensor_count(gguf_file_t f) { return f ? (int64_t)f->tensors.size() : GGUF_ERR_INVALID_ARG; }

int gguf_file_tensor_info(gguf_file_t f, int64_t index, char* name, size_t name_cap, int* type, int* n_dims,
                          int64_t dims[4], uint64_t* file_offset, uint64_t* nbytes) {
    if (!f || index < 0 || index >= (int64_t)f->tensors.size()) return GGUF_ERR_INVALID_ARG;
    const Tensor& t = f->tensors[(size_t)index];
    if (name) {
        if (name_cap < t.name.size() + 1) return GGUF_ERR_WORKSPACE;
        std::memcpy(name, t.name.c_str(), t.name.size() + 1);
    }
    if (type) *type = (int)t.type;
    if (n_dims) *n_dims = (int)t.n_dims;
    if (dims)
        for (int d = 0; d < 4; ++d) dims[d] = t.dims[d];
    if (file_offset) *file_offset = t.offset;
    if (nbytes) *nbytes = t.nbytes;
    return GGUF_OK;
}

int64_t gguf_file_find_tensor(gguf_file_t f, const char* name) {
    if (!f || !name) return GGUF_ERR_INVALID_ARG;
    for (size_t i = 0; i < f->tensors.size(); ++i)
        if (f->tensors[i].name == name) return (int64_t)i;
    return GGUF_ERR_NOT_FOUND;
}

int gguf_file_read_tensor(gguf_file_t f, int64_t index, void* host_dst, size_t dst_bytes) {
    if (!f || !host_dst || index < 0 || index >= (int64_t)f->tensors.size()) return GGUF_ERR_INVALID_ARG;
    const Tensor& t = f->tensors[(size_t)index];
    if (t.nbytes == 0) return GGUF_ERR_UNSUPPORTED;
    if (dst_bytes < t.nbytes) return GGUF_ERR_WORKSPACE;
    std::memcpy(host_dst, f->map + t.offset, (size_t)t.nbytes);
    return GGUF_OK;
}

int gguf_file_tensor_as_weight(gguf_file_t f, int64_t index, int* qtype, int64_t* N, int64_t* K) {
    if (!f || index < 0 || index >= (int64_t)f->tensors.size()) return GGUF_ERR_INVALID_ARG;
    const Tensor& t = f->tensors[(size_t)index];
    switch (t.type) {
        case GGUF_Q4_0: case GGUF_Q4_1: case GGUF_Q5_0: case GGUF_Q5_1: case GGUF_Q8_0:
        case GGUF_Q2_K: case GGUF_Q3_K: case GGUF_Q4_K: case GGUF_Q5_K: case GGUF_Q6_K: break;
        default: return GGUF_ERR_UNSUPPORTED;
    }
    if (t.dims[2] != 1 || t.dims[3] != 1) return GGUF_ERR_UNSUPPORTED;
    if (qtype) *qtype = (int)t.type;
    if (K) *K = t.dims[0];
    if (N) *N = t.dims[1];
    return GGUF_OK;
}

int64_t gguf_file_kv_count(gguf_file_t f) { return f ? (int64_t)f->kv.size() : GGUF_ERR_INVALID_ARG; }

int gguf_file_kv_key(gguf_file_t f, int64_t index, char* key, size_t cap, int* value_type) {
    if (!f || index < 0 || index >= (int64_t)f->kv.size()) return GGUF_ERR_INVALID_ARG;
    const KV& e = f->kv[(size_t)index];
    if (key) {
        if (cap < e.key.size() + 1) return GGUF_ERR_WORKSPACE;
        std::memcpy(key, e.key.c_str(), e.key.size() + 1);
    }
    if (value_type) *value_type = (int)e.v.type;
    return GGUF_OK;
}

int gguf_file_get_int(gguf_file_t f, const char* key, int64_t* out) {
    if (!f || !key || !out) return GGUF_ERR_INVALID_ARG;
    const KV* e = find_kv(f, key);
    if (!e) return GGUF_ERR_NOT_FOUND;
    const uint8_t* p = f->map + e->v.pos;
    switch (e->v.type) {
        case VT_U8: *out = p[0]; break;
        case VT_I8: *out = (int8_t)p[0]; break;
        case VT_BOOL: *out = p[0] != 0; break;
        case VT_U16: { uint16_t v; std::memcpy(&v, p, 2); *out = v; break; }
        case VT_I16: { int16_t v; std::memcpy(&v, p, 2); *out = v; break; }
        case VT_U32: { uint32_t v; std::memcpy(&v, p, 4); *out = v; break; }
        case VT_I32: { int32_t v; std::memcpy(&v, p, 4); *out = v; break; }
        case VT_U64: { uint64_t v; std::memcpy(&v, p, 8); if (v > (uint64_t)INT64_MAX) return GGUF_ERR_UNSUPPORTED; *out = (int64_t)v; break; }
        case VT_I64: { int64_t v; std::memcpy(&v, p, 8); *out = v; break; }
        default: return GGUF_ERR_UNSUPPORTED;
    }
    return GGUF_OK;
}

int gguf_file_get_float(gguf_file_t f, const char* key, double* out) {
    if (!f || !key || !out) return GGUF_ERR_INVALID_ARG;
    const KV* e = find_kv(f, key);
    if (!e) return GGUF_ERR_NOT_FOUND;
    const uint8_t* p = f->map + e->v.pos;
    if (e->v.type == VT_F32) { float v; std::memcpy(&v, p, 4); *out = v; return GGUF_OK; }
    if (e->v.type == VT_F64) { double v; std::memcpy(&v, p, 8); *out = v; return GGUF_OK; }
    int64_t i = 0;
    const int rc = gguf_file_get_int(f, key, &i);
    if (rc != GGUF_OK) return rc;
    *out = (double)i;
    return GGUF_OK;
}

int gguf_file_get_string(gguf_file_t f, const char* key, char* buf, size_t cap, size_t* len) {
    if (!f || !key) return GGUF_ERR_INVALID_ARG;
    const KV* e = find_kv(f, key);
    if (!e) return GGUF_ERR_NOT_FOUND;
    if (e->v.type != VT_STRING) return GGUF_ERR_UNSUPPORTED;
    if (len) *len = (size_t)e->v.count;
    if (buf) {
        if (cap < e->v.count + 1) return GGUF_ERR_WORKSPACE;
        std::memcpy(buf, f->map + e->v.pos, (size_t)e->v.count);
        buf[e->v.count] = '\0';
    }
    return GGUF_OK;
}

int gguf_file_get_array(gguf_file_t f, const char* key, int* elem_type, int64_t* count, void* dst, size_t cap) {
    if (!f || !key) return GGUF_ERR_INVALID_ARG;
    const KV* e = find_kv(f, key);
    if (!e) return GGUF_ERR_NOT_FOUND;
    if (e->v.type != VT_ARRAY) return GGUF_ERR_UNSUPPORTED;
    if (elem_type) *elem_type = (int)e->v.elem;
    if (count) *count = (int64_t)e->v.count;
    if (dst) {
        const int es = scalar_size(e->v.elem);
        if (es == 0) return GGUF_ERR_UNSUPPORTED;   // string arrays: element sizes vary
        if (cap < e->v.count * (uint64_t)es) return GGUF_ERR_WORKSPACE;
        std::memcpy(dst, f->map + e->v.pos, (size_t)(e->v.count * (uint64_t)es));
    }
    return GGUF_OK;
}

}  // extern "C"

// The .trit v1 container reader: parse and validate ("The .trit format,
// version 1" -- 2 File layout, 2.1, 2.2, 2.3, 2.4, 4 Validation), then hand
// out the tensors' bytes where they lie -- in the memory map -- and upload a
// ternary tensor to the device as one copy of those bytes.
//
// Every multi-byte field is assembled from bytes (little-endian by definition,
// independent of the host's byte order); every read is bounds-checked against
// the data length, so a truncated or hostile file can only produce a status.
#include <cuda_runtime.h>
#include <fcntl.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>
#include <sys/mman.h>
#include <sys/stat.h>
#include <unistd.h>

#include <algorithm>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include "trit_file.h"

namespace {

constexpr uint64_t kMaxConfig = 16ull * 1024 * 1024;
constexpr uint64_t kMaxTensors = 1048576;
constexpr uint32_t kMaxName = 1024;
constexpr uint64_t kFnvBasis = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

struct Record {
    uint64_t name_at;      // byte offset of the name in the file
    uint32_t name_len;
    uint32_t dtype, ndim;
    uint32_t dims[4];
    float scale;
    uint64_t offset, byte_len;
    bool prod_ok;          // the product of dims fits 64 bits
    uint64_t prod;
};

struct Fail {
    trit_file_status st;
    std::string msg;
};

void put_msg(char *msg, size_t len, const std::string &s) {
    if (!msg || len == 0) return;
    const size_t n = s.size() < len - 1 ? s.size() : len - 1;
    memcpy(msg, s.data(), n);
    msg[n] = '\0';
}

std::string fmt(const char *f, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, f);
    vsnprintf(buf, sizeof buf, f, ap);
    va_end(ap);
    return buf;
}

bool valid_utf8(const uint8_t *p, uint64_t n) {
    uint64_t i = 0;
    while (i < n) {
        const uint8_t c = p[i];
        uint32_t need, cp;
        if (c < 0x80) {
            ++i;
            continue;
        } else if ((c & 0xE0) == 0xC0) {
            need = 1;
            cp = c & 0x1F;
        } else if ((c & 0xF0) == 0xE0) {
            need = 2;
            cp = c & 0x0F;
        } else if ((c & 0xF8) == 0xF0) {
            need = 3;
            cp = c & 0x07;
        } else {
            return false;
        }
        if (n - i - 1 < need) return false;   // the sequence runs past the end
        for (uint32_t k = 1; k <= need; ++k) {
            const uint8_t d = p[i + k];
            if ((d & 0xC0) != 0x80) return false;
            cp = (cp << 6) | (d & 0x3F);
        }
        // shortest form, no surrogates, at most U+10FFFF
        if ((need == 1 && cp < 0x80) || (need == 2 && cp < 0x800) || (need == 3 && cp < 0x10000) ||
            (cp >= 0xD800 && cp <= 0xDFFF) || cp > 0x10FFFF)
            return false;
        i += need + 1;
    }
    return true;
}

// Bounds-checked little-endian cursor over the file's bytes.
struct Cursor {
    const uint8_t *p;
    uint64_t len, pos;
    bool take(uint64_t n, const uint8_t **at) {
        if (n > len - pos) return false;
        *at = p + pos;
        pos += n;
        return true;
    }
    bool uint(int bytes, uint64_t *v) {
        const uint8_t *a;
        if (!take(uint64_t(bytes), &a)) return false;
        uint64_t x = 0;
        for (int i = bytes - 1; i >= 0; --i) x = (x << 8) | a[i];
        *v = x;
        return true;
    }
};

float f32_from_bits(uint32_t b) {
    float f;
    memcpy(&f, &b, 4);
    return f;
}

uint64_t load_u64(const uint8_t *a) {
    uint64_t x = 0;
    for (int i = 7; i >= 0; --i) x = (x << 8) | a[i];
    return x;
}

}  // namespace

struct trit_file {
    const uint8_t *data = nullptr;
    uint64_t len = 0;
    void *map = nullptr;        // owned mapping (trit_file_open), else NULL
    size_t map_len = 0;
    uint64_t payload_hash = 0;
    uint64_t config_at = 0;
    uint32_t config_len = 0;
    uint64_t payload_start = 0;
    std::vector<Record> recs;
    std::vector<uint32_t> by_name;   // record indices sorted by name bytes

    std::string name(uint32_t i) const {
        return std::string(reinterpret_cast<const char *>(data + recs[i].name_at), recs[i].name_len);
    }
};

namespace {

// Checks 1-16 in the order stated in trit_file.h.
bool parse(trit_file &f, Fail &fail) {
    Cursor c{f.data, f.len, 0};
    auto trunc = [&](const char *what) {
        fail = {TRIT_F_TRUNCATED, fmt("truncated file: %s lies past byte %llu", what,
                                      (unsigned long long)f.len)};
        return false;
    };
    const uint8_t *magic;
    if (!c.take(4, &magic)) return trunc("the magic");
    if (memcmp(magic, "TRIT", 4) != 0) {
        fail = {TRIT_F_MAGIC, "not a .trit file: the first four bytes are not \"TRIT\""};
        return false;
    }
    uint64_t version, flags, hash, config_len, count;
    if (!c.uint(4, &version)) return trunc("version");
    if (version == 0) {
        fail = {TRIT_F_V0, "a version 0 file (2-bit interleaved codes) is not read: convert the "
                           "source checkpoint again, or upgrade the file with the converter"};
        return false;
    }
    if (version > 1) {
        fail = {TRIT_F_VERSION, fmt("version %llu is not supported (this reader reads version 1)",
                                    (unsigned long long)version)};
        return false;
    }
    if (!c.uint(4, &flags)) return trunc("header_flags");
    if (flags != 0) {
        fail = {TRIT_F_HEADER_FLAGS, fmt("unknown header flags 0x%llx", (unsigned long long)flags)};
        return false;
    }
    if (!c.uint(8, &hash)) return trunc("payload_hash");
    f.payload_hash = hash;
    if (!c.uint(4, &config_len)) return trunc("config_len");
    if (config_len > kMaxConfig) {
        fail = {TRIT_F_CONFIG, fmt("config_len %llu exceeds 16 MiB", (unsigned long long)config_len)};
        return false;
    }
    const uint8_t *config;
    if (!c.take(config_len, &config)) return trunc("the config");
    if (!valid_utf8(config, config_len)) {
        fail = {TRIT_F_CONFIG, "the config is not valid UTF-8"};
        return false;
    }
    f.config_at = uint64_t(config - f.data);
    f.config_len = uint32_t(config_len);
    if (!c.uint(4, &count)) return trunc("tensor_count");
    if (count > kMaxTensors) {
        fail = {TRIT_F_RECORD, fmt("tensor_count %llu exceeds 1048576", (unsigned long long)count)};
        return false;
    }
    // a record takes at least 35 bytes: never reserve more than the data can hold
    const uint64_t fit = (f.len - c.pos) / 35;
    f.recs.reserve(size_t(count < fit ? count : fit));
    for (uint64_t t = 0; t < count; ++t) {
        Record r{};
        uint64_t v;
        if (!c.uint(2, &v)) return trunc("a tensor record");
        if (v == 0 || v > kMaxName) {
            fail = {TRIT_F_NAME, fmt("tensor %llu: name_len %llu is outside 1..1024",
                                     (unsigned long long)t, (unsigned long long)v)};
            return false;
        }
        r.name_len = uint32_t(v);
        const uint8_t *name;
        if (!c.take(v, &name)) return trunc("a tensor name");
        if (!valid_utf8(name, v)) {
            fail = {TRIT_F_NAME, fmt("tensor %llu: the name is not valid UTF-8", (unsigned long long)t)};
            return false;
        }
        r.name_at = uint64_t(name - f.data);
        const std::string nm(reinterpret_cast<const char *>(name), r.name_len);
        uint64_t dtype, ndim, res0, res1, dim, scale_bits, tflags;
        if (!c.uint(1, &dtype) || !c.uint(1, &ndim) || !c.uint(1, &res0) || !c.uint(1, &res1))
            return trunc("a tensor record");
        if (ndim < 1 || ndim > 4) {
            fail = {TRIT_F_RECORD, fmt("tensor '%s': ndim %llu is outside 1..4", nm.c_str(),
                                       (unsigned long long)ndim)};
            return false;
        }
        r.dtype = uint32_t(dtype);
        r.ndim = uint32_t(ndim);
        for (uint64_t d = 0; d < ndim; ++d) {
            if (!c.uint(4, &dim)) return trunc("a tensor's dims");
            r.dims[d] = uint32_t(dim);
        }
        if (!c.uint(4, &scale_bits) || !c.uint(4, &tflags) || !c.uint(8, &r.offset) ||
            !c.uint(8, &r.byte_len))
            return trunc("a tensor record");
        r.scale = f32_from_bits(uint32_t(scale_bits));
        if (dtype > 2 || res0 != 0 || res1 != 0 || tflags != 0) {
            fail = {TRIT_F_RECORD,
                    fmt("tensor '%s': dtype %llu, reserved bytes %llu/%llu, flags 0x%llx (dtype "
                        "must be 0..2, the others 0)",
                        nm.c_str(), (unsigned long long)dtype, (unsigned long long)res0,
                        (unsigned long long)res1, (unsigned long long)tflags)};
            return false;
        }
        unsigned __int128 prod = 1;
        r.prod_ok = true;
        for (uint32_t d = 0; d < r.ndim; ++d) {
            prod *= r.dims[d];
            if (prod >> 64) r.prod_ok = false;
        }
        if (!r.prod_ok) {
            fail = {TRIT_F_SHAPE, fmt("tensor '%s': the product of its dims overflows 64 bits",
                                      nm.c_str())};
            return false;
        }
        r.prod = uint64_t(prod);
        if (!isfinite(r.scale) || !(r.scale > 0.0f)) {
            fail = {TRIT_F_SCALE, fmt("tensor '%s': scale %g is not finite and positive", nm.c_str(),
                                      double(r.scale))};
            return false;
        }
        if (r.offset % 64 != 0) {
            fail = {TRIT_F_ALIGN, fmt("tensor '%s': offset %llu is not a multiple of 64", nm.c_str(),
                                      (unsigned long long)r.offset)};
            return false;
        }
        f.recs.push_back(r);
    }
    const uint64_t end = c.pos;
    const uint64_t ps = (end + 63) / 64 * 64;
    if (ps > f.len) return trunc("payload_start");
    f.payload_start = ps;
    const uint64_t plen = f.len - ps;
    for (uint32_t i = 0; i < f.recs.size(); ++i) {
        const Record &r = f.recs[i];
        if (r.offset > plen || r.byte_len > plen - r.offset) {
            fail = {TRIT_F_EXTENT, fmt("tensor '%s': bytes %llu..+%llu lie past the payload "
                                       "(%llu bytes)",
                                       f.name(i).c_str(), (unsigned long long)r.offset,
                                       (unsigned long long)r.byte_len, (unsigned long long)plen)};
            return false;
        }
        if (r.dtype == TRIT_DTYPE_TRIT) {
            if (r.ndim != 2) {
                fail = {TRIT_F_TRIT_NDIM, fmt("ternary tensor '%s' has %u dims, not 2",
                                              f.name(i).c_str(), r.ndim)};
                return false;
            }
            const unsigned __int128 want =
                (unsigned __int128)r.dims[0] * ((uint64_t(r.dims[1]) + 63) / 64) * 16;
            if (want != r.byte_len) {
                fail = {TRIT_F_TRIT_BYTES, fmt("ternary tensor '%s': byte_len %llu != rows x "
                                               "beats_per_row x 16",
                                               f.name(i).c_str(), (unsigned long long)r.byte_len)};
                return false;
            }
        } else {
            const unsigned __int128 want =
                (unsigned __int128)r.prod * (r.dtype == TRIT_DTYPE_F32 ? 4 : 2);
            if (want != r.byte_len) {
                fail = {TRIT_F_DENSE_BYTES, fmt("dense tensor '%s': byte_len %llu != elements x "
                                                "element size",
                                                f.name(i).c_str(), (unsigned long long)r.byte_len)};
                return false;
            }
        }
    }
    f.by_name.resize(f.recs.size());
    for (uint32_t i = 0; i < f.recs.size(); ++i) f.by_name[i] = i;
    auto less = [&](uint32_t a, uint32_t b) {
        const Record &x = f.recs[a], &y = f.recs[b];
        const int c2 = memcmp(f.data + x.name_at, f.data + y.name_at,
                              x.name_len < y.name_len ? x.name_len : y.name_len);
        return c2 != 0 ? c2 < 0 : x.name_len < y.name_len;
    };
    std::sort(f.by_name.begin(), f.by_name.end(), less);
    for (size_t k = 1; k < f.by_name.size(); ++k) {
        if (!less(f.by_name[k - 1], f.by_name[k])) {
            fail = {TRIT_F_NAME, fmt("duplicate tensor name '%s'", f.name(f.by_name[k]).c_str())};
            return false;
        }
    }
    std::vector<std::pair<uint64_t, uint64_t>> ext;
    for (const Record &r : f.recs)
        if (r.byte_len > 0) ext.push_back({r.offset, r.offset + r.byte_len});
    std::sort(ext.begin(), ext.end());
    for (size_t k = 1; k < ext.size(); ++k) {
        if (ext[k].first < ext[k - 1].second) {
            fail = {TRIT_F_OVERLAP, fmt("two tensors' payload extents overlap at payload byte %llu",
                                        (unsigned long long)ext[k].first)};
            return false;
        }
    }
    return true;
}

trit_file_status open_common(trit_file *f, trit_file **out, char *msg, size_t msg_len) {
    Fail fail{TRIT_F_OK, ""};
    if (!parse(*f, fail)) {
        put_msg(msg, msg_len, fail.msg);
        trit_file_close(f);
        return fail.st;
    }
    put_msg(msg, msg_len, "");
    *out = f;
    return TRIT_F_OK;
}

}  // namespace

extern "C" {

TRIT_API uint64_t trit_fnv1a64(const uint8_t *data, uint64_t len) {
    uint64_t h = kFnvBasis;
    for (uint64_t i = 0; i < len; ++i) {
        h ^= data[i];
        h *= kFnvPrime;
    }
    return h;
}

TRIT_API trit_file_status trit_file_open_memory(const uint8_t *data, uint64_t len, trit_file **out,
                                                char *msg, size_t msg_len) {
    if (!out || (!data && len > 0)) {
        put_msg(msg, msg_len, "NULL argument");
        return TRIT_F_ARG;
    }
    *out = nullptr;
    trit_file *f = new (std::nothrow) trit_file;
    if (!f) return TRIT_F_NOMEM;
    f->data = data;
    f->len = len;
    return open_common(f, out, msg, msg_len);
}

TRIT_API trit_file_status trit_file_open(const char *path, trit_file **out, char *msg,
                                         size_t msg_len) {
    if (!out || !path) {
        put_msg(msg, msg_len, "NULL argument");
        return TRIT_F_ARG;
    }
    *out = nullptr;
    const int fd = open(path, O_RDONLY);
    if (fd < 0) {
        put_msg(msg, msg_len, fmt("cannot open %s", path));
        return TRIT_F_IO;
    }
    struct stat sb;
    if (fstat(fd, &sb) != 0) {
        close(fd);
        put_msg(msg, msg_len, fmt("cannot stat %s", path));
        return TRIT_F_IO;
    }
    void *map = nullptr;
    const size_t n = size_t(sb.st_size);
    if (n > 0) {
        map = mmap(nullptr, n, PROT_READ, MAP_PRIVATE, fd, 0);
        if (map == MAP_FAILED) {
            close(fd);
            put_msg(msg, msg_len, fmt("cannot map %s", path));
            return TRIT_F_IO;
        }
    }
    close(fd);
    trit_file *f = new (std::nothrow) trit_file;
    if (!f) {
        if (map) munmap(map, n);
        return TRIT_F_NOMEM;
    }
    f->data = static_cast<const uint8_t *>(map);
    f->len = n;
    f->map = map;
    f->map_len = n;
    return open_common(f, out, msg, msg_len);
}

TRIT_API void trit_file_close(trit_file *f) {
    if (!f) return;
    if (f->map) munmap(f->map, f->map_len);
    delete f;
}

TRIT_API trit_file_status trit_file_verify(const trit_file *f, char *msg, size_t msg_len) {
    if (!f) {
        put_msg(msg, msg_len, "NULL argument");
        return TRIT_F_ARG;
    }
    for (uint32_t i = 0; i < f->recs.size(); ++i) {
        const Record &r = f->recs[i];
        if (r.dtype != TRIT_DTYPE_TRIT) continue;
        const uint64_t rows = r.dims[0], cols = r.dims[1], bpr = (cols + 63) / 64;
        const uint64_t tail = cols % 64 == 0 ? ~uint64_t(0) : (uint64_t(1) << (cols % 64)) - 1;
        const uint8_t *base = f->data + f->payload_start + r.offset;
        for (uint64_t row = 0; row < rows; ++row) {
            const uint8_t *rp = base + row * bpr * 16;
            for (uint64_t b = 0; b < bpr; ++b) {
                const uint64_t both = load_u64(rp + b * 16) & load_u64(rp + b * 16 + 8);
                if (both) {
                    int k = 0;
                    while (!((both >> k) & 1)) ++k;
                    put_msg(msg, msg_len,
                            fmt("P1: tensor '%s' row %llu beat %llu column %llu has both bits set",
                                f->name(i).c_str(), (unsigned long long)row, (unsigned long long)b,
                                (unsigned long long)(b * 64 + k)));
                    return TRIT_F_P1;
                }
            }
            const uint8_t *last = rp + (bpr - 1) * 16;
            if (bpr > 0 && ((load_u64(last) | load_u64(last + 8)) & ~tail)) {
                put_msg(msg, msg_len, fmt("P2: tensor '%s' row %llu has a padding bit set",
                                          f->name(i).c_str(), (unsigned long long)row));
                return TRIT_F_P2;
            }
        }
    }
    if (f->payload_hash != 0) {
        const uint64_t h = trit_fnv1a64(f->data + f->payload_start, f->len - f->payload_start);
        if (h != f->payload_hash) {
            put_msg(msg, msg_len, fmt("payload hash 0x%016llx does not match the stored 0x%016llx",
                                      (unsigned long long)h, (unsigned long long)f->payload_hash));
            return TRIT_F_HASH;
        }
    }
    put_msg(msg, msg_len, "");
    return TRIT_F_OK;
}

TRIT_API uint32_t trit_file_tensor_count(const trit_file *f) {
    return f ? uint32_t(f->recs.size()) : 0;
}

TRIT_API trit_file_status trit_file_tensor(const trit_file *f, uint32_t i, trit_tensor_info *info) {
    if (!f || !info || i >= f->recs.size()) return TRIT_F_ARG;
    const Record &r = f->recs[i];
    memset(info, 0, sizeof *info);
    info->name = reinterpret_cast<const char *>(f->data + r.name_at);
    info->name_len = r.name_len;
    info->dtype = r.dtype;
    info->ndim = r.ndim;
    for (uint32_t d = 0; d < r.ndim; ++d) info->dims[d] = r.dims[d];
    info->scale = r.scale;
    info->offset = r.offset;
    info->byte_len = r.byte_len;
    info->data = f->data + f->payload_start + r.offset;
    return TRIT_F_OK;
}

TRIT_API int64_t trit_file_find(const trit_file *f, const char *name, uint32_t name_len) {
    if (!f || (!name && name_len)) return -1;
    size_t lo = 0, hi = f->by_name.size();
    while (lo < hi) {
        const size_t mid = (lo + hi) / 2;
        const Record &r = f->recs[f->by_name[mid]];
        int c = memcmp(f->data + r.name_at, name, r.name_len < name_len ? r.name_len : name_len);
        if (c == 0) c = r.name_len < name_len ? -1 : (r.name_len > name_len ? 1 : 0);
        if (c == 0) return int64_t(f->by_name[mid]);
        if (c < 0) lo = mid + 1;
        else hi = mid;
    }
    return -1;
}

TRIT_API const uint8_t *trit_file_config(const trit_file *f, uint32_t *len) {
    if (!f) return nullptr;
    if (len) *len = f->config_len;
    return f->data + f->config_at;
}

TRIT_API uint64_t trit_file_payload_hash(const trit_file *f) { return f ? f->payload_hash : 0; }
TRIT_API uint64_t trit_file_payload_start(const trit_file *f) { return f ? f->payload_start : 0; }
TRIT_API uint64_t trit_file_payload_len(const trit_file *f) {
    return f ? f->len - f->payload_start : 0;
}

TRIT_API trit_status trit_file_upload(const trit_file *f, uint32_t i, void *dst,
                                      trit_stream_t stream) {
    if (!f || !dst || i >= f->recs.size()) return TRIT_E_ARG;
    const Record &r = f->recs[i];
    if (r.dtype == TRIT_DTYPE_TRIT && (reinterpret_cast<uintptr_t>(dst) & 15) != 0) return TRIT_E_ARG;
    if (r.byte_len == 0) return TRIT_OK;
    const cudaError_t e = cudaMemcpyAsync(dst, f->data + f->payload_start + r.offset,
                                          size_t(r.byte_len), cudaMemcpyHostToDevice,
                                          reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TRIT_OK : TRIT_E_CUDA;
}

}  // extern "C"

/*
 * trit_file.h -- C ABI of libtrit's .trit v1 container reader ("The .trit
 * format, version 1" -- 2 File layout, 2.1 Header fields, 2.2 Tensor record,
 * 2.3 Ternary payload, 2.4 Dense payload, 4 Validation).
 *
 * A .trit file holds a header, the source config.json, a table of tensor
 * records and a payload whose start is a multiple of 64 bytes.  Ternary
 * tensors are stored exactly as the kernels of trit.h read them (N rows x
 * ceil(K/64) beats x 16 bytes), so a tensor is uploaded to the device as one
 * copy of its bytes, never repacked.
 *
 * Opening runs the header checks (the page's checks 1-16, O(tensor_count));
 * trit_file_verify runs the payload checks (17-19, O(file size)) on the host;
 * a tensor already on the device can instead be checked with trit_verify.
 * Every rejection returns the number of the failed check as its status and a
 * message naming the field, tensor, row, beat or column involved.
 *
 * Readings where the page is silent:
 *   - a read past the end of the data, including a file shorter than the
 *     4-byte magic, is check 5;
 *   - tensor_count > 1,048,576 is reported as check 8;
 *   - a tensor name that is not valid UTF-8 is check 7;
 *   - the padding before payload_start is located, not inspected;
 *   - order: header fields as read (1, 2/3, 4, 6, count); each record as read:
 *     name (7), ndim (8), then dtype / reserved / flags (8), shape product (9),
 *     scale (10), offset alignment (11); then per record in file order 12,
 *     14, 15/16; then duplicate names (7); then overlapping extents (13).
 *     Verification: ternary tensors in record order, rows in order, a row's
 *     P1 on every beat (17) before its P2 (18), then the hash (19);
 *   - the hash is standard FNV-1a-64 (basis 0xcbf29ce484222325, prime
 *     0x100000001b3) as section 2 names it; a stored hash of 0 is "absent" and
 *     not checked.  The worked example of section 3 stores a value made with
 *     the prime 0x1000000001b3, so it fails check 19 here.
 */
#ifndef TRIT_FILE_H
#define TRIT_FILE_H

#include <stddef.h>
#include <stdint.h>

#include "trit.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Status of the container calls: 0, or the number of the failed check. */
typedef enum trit_file_status {
    TRIT_F_OK = 0,
    TRIT_F_MAGIC = 1,          /* not a .trit file */
    TRIT_F_V0 = 2,             /* version 0 (2-bit interleaved codes): re-convert or upgrade */
    TRIT_F_VERSION = 3,        /* version > 1 */
    TRIT_F_HEADER_FLAGS = 4,   /* header_flags != 0 */
    TRIT_F_TRUNCATED = 5,      /* a field lies past the end of the data */
    TRIT_F_CONFIG = 6,         /* config_len > 16 MiB or config not UTF-8 */
    TRIT_F_NAME = 7,           /* name_len 0 or > 1024, not UTF-8, or duplicate */
    TRIT_F_RECORD = 8,         /* dtype, ndim, reserved bytes, flags or tensor_count */
    TRIT_F_SHAPE = 9,          /* product of dims overflows 64 bits */
    TRIT_F_SCALE = 10,         /* scale not finite or <= 0 */
    TRIT_F_ALIGN = 11,         /* offset % 64 != 0 */
    TRIT_F_EXTENT = 12,        /* offset + byte_len past the end of the payload */
    TRIT_F_OVERLAP = 13,       /* two tensors' payload extents overlap */
    TRIT_F_TRIT_NDIM = 14,     /* ternary tensor that is not 2-D */
    TRIT_F_TRIT_BYTES = 15,    /* ternary byte_len != rows * ceil(cols/64) * 16 */
    TRIT_F_DENSE_BYTES = 16,   /* dense byte_len != prod(dims) * element size */
    TRIT_F_P1 = 17,            /* a beat with a bit set in both planes */
    TRIT_F_P2 = 18,            /* a padding bit past cols is set */
    TRIT_F_HASH = 19,          /* payload_hash mismatch */
    TRIT_F_IO = 32,            /* the file could not be opened or mapped */
    TRIT_F_ARG = 33,           /* NULL argument or index out of range */
    TRIT_F_NOMEM = 34          /* host allocation failed */
} trit_file_status;

typedef enum trit_dtype { TRIT_DTYPE_F32 = 0, TRIT_DTYPE_TRIT = 1, TRIT_DTYPE_BF16 = 2 } trit_dtype;

/* An opened, header-validated file (opaque; one per trit_file_open*). */
typedef struct trit_file trit_file;

/* One tensor record.  name points into the file's bytes (not NUL-terminated:
 * name_len bytes); data points at the tensor's payload bytes on the host. */
typedef struct trit_tensor_info {
    const char *name;
    uint32_t name_len;
    uint32_t dtype;          /* trit_dtype */
    uint32_t ndim;           /* 1..4 */
    uint32_t dims[4];        /* outermost first; unused entries 0 */
    float scale;             /* dequantisation factor (ternary), 1.0 for dense */
    uint32_t reserved;       /* 0 */
    uint64_t offset;         /* relative to payload_start, multiple of 64 */
    uint64_t byte_len;
    const uint8_t *data;     /* host address of the payload bytes */
} trit_tensor_info;

/* Map the file at `path` read-only and run checks 1-16.  On success *out owns
 * the mapping (release with trit_file_close).  On failure *out is NULL and,
 * when msg is not NULL, a NUL-terminated explanation of at most msg_len bytes
 * is written there. */
TRIT_API trit_file_status trit_file_open(const char *path, trit_file **out, char *msg,
                                         size_t msg_len);

/* The same on `len` bytes the caller keeps alive (and unchanged) until
 * trit_file_close. */
TRIT_API trit_file_status trit_file_open_memory(const uint8_t *data, uint64_t len, trit_file **out,
                                                char *msg, size_t msg_len);

/* Release the file (and the mapping of trit_file_open).  NULL is ignored. */
TRIT_API void trit_file_close(trit_file *f);

/* Checks 17-19 on the host (P1 on every beat, P2 on every row's last beat, the
 * payload hash when stored).  The first violation decides the status. */
TRIT_API trit_file_status trit_file_verify(const trit_file *f, char *msg, size_t msg_len);

TRIT_API uint32_t trit_file_tensor_count(const trit_file *f);

/* Record i (file order) into *info. */
TRIT_API trit_file_status trit_file_tensor(const trit_file *f, uint32_t i, trit_tensor_info *info);

/* Index of the tensor whose name is the name_len bytes at name, or -1. */
TRIT_API int64_t trit_file_find(const trit_file *f, const char *name, uint32_t name_len);

/* The embedded config.json: *len bytes at the returned address (host). */
TRIT_API const uint8_t *trit_file_config(const trit_file *f, uint32_t *len);

/* The stored payload_hash (0 = absent), payload_start and payload length. */
TRIT_API uint64_t trit_file_payload_hash(const trit_file *f);
TRIT_API uint64_t trit_file_payload_start(const trit_file *f);
TRIT_API uint64_t trit_file_payload_len(const trit_file *f);

/* Standard FNV-1a-64 of len bytes. */
TRIT_API uint64_t trit_fnv1a64(const uint8_t *data, uint64_t len);

/* Copy tensor i's payload bytes, unchanged, to the DEVICE address dst
 * (byte_len bytes, caller-owned; 16-byte aligned for ternary tensors so that
 * the kernels of trit.h can read them) with cudaMemcpyAsync on `stream`.  The
 * copy reads the host bytes asynchronously: keep the file open until the
 * stream has synchronised.  Returns TRIT_OK, TRIT_E_ARG (NULL, index out of
 * range, misaligned ternary destination) or TRIT_E_CUDA. */
TRIT_API trit_status trit_file_upload(const trit_file *f, uint32_t i, void *dst,
                                      trit_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TRIT_FILE_H */

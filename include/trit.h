/*
 * trit.h -- C ABI of libtrit: ternary select-accumulate matrix-vector and
 * matrix-matrix products over .trit v1 bit planes, on NVIDIA GB300 (sm_103a).
 *
 * For an output row r the product is
 *     y_r = sum_{c : W[r][c] = +1} x_c  -  sum_{c : W[r][c] = -1} x_c,
 * with no multiplications ("Tritium: One Weight Format for Ternary Inference
 * on Commodity CPUs and Multiplier-Free Hardware" -- Introduction, Eq. 3;
 * "The .trit format, version 1" -- 1 Why bit planes).
 *
 * Layouts
 *   planes   The .trit v1 ternary payload ("The .trit format, version 1" --
 *            2.3): N rows x B = ceil(K/64) beats x 16 bytes, row-major.  Beat b
 *            of row r is at byte (r*B + b)*16: bytes 0..8 a little-endian u64
 *            `pos` (bit k set <=> W[r][64b+k] = +1), bytes 8..16 `neg`
 *            (bit k set <=> W[r][64b+k] = -1).  Both bits set is illegal (P1);
 *            padding bits past column K must be clear (P2).
 *   x_i8     M activation rows of int8, row stride K_pad = 64*B bytes; only
 *            columns < K are read (the library zero-fills the tail itself).
 *   x_scale  M fp32 per-row scales, the absmax of each quantised row.
 *   y_i32    M x N int32, row-major: the exact integer products.
 *   y_f32    M x N fp32, row-major:
 *            (((float)y_i32 * w_scale) * x_scale[m]) / 127, each step rounded
 *            to nearest in fp32 ("Tritium ..." -- Why exactness, concretely:
 *            scale by each factor in turn).
 *
 * Conventions for every entry point
 *   - Data pointers are DEVICE pointers to caller-owned memory.  The library
 *     keeps no pointer after the call returns.  The only device memory it
 *     allocates is the temporary fp16 copy of the activations used by the
 *     tensor-core path of trit_gemm / trit_gemm_many (M >= 13): allocated with
 *     cudaMallocAsync on the call's stream and freed, stream-ordered, after the
 *     launches (failure returns TRIT_E_CUDA).  trit_gemm_noalloc allocates
 *     nothing (it uses a fixed buffer instead, see there).
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *     call returns without synchronising; results are valid once the stream
 *     has synchronised.
 *   - Argument errors found on the host return a nonzero trit_status and
 *     enqueue nothing.  A failed CUDA launch returns TRIT_E_CUDA
 *     (trit_last_cuda_error() names it).
 *   - Errors in the data are OR-ed by the kernels into *err_flag, a device
 *     uint32 (TRIT_ERR_* bits).  Kernels only set bits: the caller zeroes the
 *     flag before the call and reads it after the stream has synchronised.
 *   - Supported sizes: 1 <= K < 2^24 (so |y| <= 128*K fits int32),
 *     1 <= N, M <= 2^31 - 1.  No size is silently skipped; anything outside
 *     returns TRIT_E_SHAPE.
 *   - Alignment: planes and x_i8 16-byte aligned; fp32/int32 arrays 4-byte
 *     aligned.
 */
#ifndef TRIT_H
#define TRIT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define TRIT_API __declspec(dllexport)
#else
#define TRIT_API __attribute__((visibility("default")))
#endif

/* Same type as cudaStream_t; declared here so that this header needs no CUDA include. */
typedef struct CUstream_st *trit_stream_t;

typedef enum trit_status {
    TRIT_OK = 0,
    TRIT_E_ARG = 1,         /* NULL where a pointer is required, count <= 0, misalignment */
    TRIT_E_SHAPE = 2,       /* a size outside the supported range */
    TRIT_E_SCALE = 4,       /* w_scale not finite or <= 0 ("The .trit format, version 1" -- 2.2);
                               trit_gemv's by-value x_scale not finite or < 0 */
    TRIT_E_CUDA = 6,        /* a CUDA runtime call or launch failed */
    TRIT_E_DEVICE = 7,      /* the current device is not an sm_103 GPU */
    TRIT_E_SCRATCH = 8,     /* trit_gemm_noalloc: the call needs more than
                               TRIT_NOALLOC_SCRATCH_BYTES of scratch */
    TRIT_E_VALUE = 9        /* trit_bitcos_pack: a weight outside {-1, 0, +1} */
} trit_status;

/* Bits of *err_flag. */
#define TRIT_ERR_P1 1u            /* a beat with pos & neg != 0 (both bits set) */
#define TRIT_ERR_P2 2u            /* a padding bit past column K is set (trit_verify only) */
#define TRIT_ERR_NOT_TERNARY 4u   /* trit_pack saw a value outside {-1, 0, +1} */
#define TRIT_ERR_NONFINITE 8u     /* trit_quant_act saw a NaN or infinity */
#define TRIT_ERR_TIMEOUT 16u      /* a bounded wait inside a kernel gave up */

/* Most list entries one launch of the *_many calls accepts; longer lists are
 * split into consecutive launches on the same stream. */
#define TRIT_MAX_LIST_PER_LAUNCH 256

/* Human-readable name of a status code (static storage). */
TRIT_API const char *trit_status_string(trit_status s);

/* Text of the last CUDA error this thread saw inside the library, or "". */
TRIT_API const char *trit_last_cuda_error(void);

/* ABI version; bumped on any change of a signature or a layout. */
TRIT_API int32_t trit_abi_version(void);

/* Bytes of the ternary payload of an N x K matrix: N * ceil(K/64) * 16
 * ("The .trit format, version 1" -- 2.3, byte_len).  Returns -1 if N or K is
 * outside the supported range. */
TRIT_API int64_t trit_payload_bytes(int64_t N, int64_t K);

/*
 * trit_pack -- int8 ternary weights to bit planes ("The .trit format,
 * version 1" -- 2.3; "Tritium ..." -- The .trit v1 layout).
 *   w          [N][K] int8, row-major, values in {-1, 0, +1}
 *   w_scale    per-tensor dequantisation factor; must be finite and > 0
 *   planes     out: N * ceil(K/64) * 16 bytes; padding bits are written clear
 *   scale_out  out, may be NULL: receives w_scale (one fp32), the scale that
 *              travels with the planes
 *   err_flag   TRIT_ERR_NOT_TERNARY if any value is outside {-1, 0, +1}; such a
 *              weight is stored as 0
 */
TRIT_API trit_status trit_pack(const int8_t *w, int64_t N, int64_t K, float w_scale,
                               uint8_t *planes, float *scale_out, uint32_t *err_flag,
                               trit_stream_t stream);

/*
 * trit_unpack -- bit planes back to int8 ternary weights [N][K] (inverse of
 * trit_pack).  A both-bits-set position sets TRIT_ERR_P1 and is written as 0
 * ("The .trit format, version 1" -- 2.3, P1: every consumer treats it as an
 * error).
 */
TRIT_API trit_status trit_unpack(const uint8_t *planes, int64_t N, int64_t K, int8_t *w,
                                 uint32_t *err_flag, trit_stream_t stream);

/*
 * trit_verify -- check P1 on every beat and P2 on every row's last beat
 * ("The .trit format, version 1" -- 2.3 and 4, checks 17 and 18; "Tritium
 * ..." -- Invariants).  P2 uses the 64-bit tail mask
 *     tail = (K % 64 == 0) ? ~0 : (1 << (K % 64)) - 1.
 *   err_flag   TRIT_ERR_P1 and/or TRIT_ERR_P2
 *   first_bad  may be NULL; else the caller initialises it to UINT64_MAX and it
 *              receives the smallest offending bit position
 *              (r*B + b)*64 + k over both kinds -- row r, beat b, bit k.
 */
TRIT_API trit_status trit_verify(const uint8_t *planes, int64_t N, int64_t K,
                                 uint32_t *err_flag, uint64_t *first_bad,
                                 trit_stream_t stream);

/*
 * trit_quant_act -- per-token absmax int8 activation quantiser ("Tritium ..."
 * -- Numerics; the pages give no formula, this is the reading used):
 *   a = max_c |x[m][c]|;  inv = 127.0f / a (IEEE fp32 division);
 *   q = clamp(round_half_even(x * inv), -127, 127);  x_scale[m] = a.
 * a = 0 gives q = 0 and x_scale = 0.  When a < 2^-96 both x and a are first
 * multiplied by 2^96 (exact) so that 127/a stays finite.  A row holding a NaN
 * or an infinity sets TRIT_ERR_NONFINITE and is written as q = 0, x_scale = 0.
 *   x        [M][K] fp32, row-major
 *   x_i8     out: [M][K_pad], K_pad = 64*ceil(K/64); columns K..K_pad-1 = 0
 *   x_scale  out: [M] fp32
 */
TRIT_API trit_status trit_quant_act(const float *x, int64_t M, int64_t K, int8_t *x_i8,
                                    float *x_scale, uint32_t *err_flag, trit_stream_t stream);

/*
 * trit_gemm -- y = W x for M activation rows (layouts above).  Integer
 * accumulation is exact (int32; every kernel gives identical bits, "Tritium
 * ..." -- CPU kernels, Verification).  The kernel is chosen by M: one row per
 * pass for M = 1, beats reused across up to 8 rows held in registers for
 * 2 <= M <= 12, and tensor cores with planes expanded to +-1 in shared memory
 * for M >= 13 (K < 131072; longer rows stay on the integer path): 128-row
 * weight tiles against all M rows (rounded up to 16) for M <= 128, 256 x 256
 * tiles on pairs of SMs above.
 *   w_scale   finite, > 0
 *   y_i32, y_f32  outputs, either may be NULL (not both)
 *   err_flag  TRIT_ERR_P1 if any beat has both bits set; the outputs of a row
 *             holding such a beat are unspecified, all other rows are exact.
 */
TRIT_API trit_status trit_gemm(const uint8_t *planes, float w_scale, const int8_t *x_i8,
                               const float *x_scale, int64_t M, int64_t N, int64_t K,
                               int32_t *y_i32, float *y_f32, uint32_t *err_flag,
                               trit_stream_t stream);

/*
 * trit_gemv -- one activation row (M = 1) with its scale passed BY VALUE:
 *     y_i32[r] = sum_{W[r][c] = +1} x_c - sum_{W[r][c] = -1} x_c,
 *     y_f32[r] = (((float)y_i32[r] * w_scale) * x_scale) / 127
 * ("Tritium ..." -- Introduction, Eq. 3; Why exactness, concretely).  The
 * results are bit-identical to trit_gemm with M = 1 and a device scale holding
 * the same value; use trit_gemm (M = 1) when the scale lives on the device, as
 * it does straight after trit_quant_act, to avoid reading it back to the host.
 *   x_i8      [K_pad] int8, device, 16-byte aligned
 *   x_scale   host fp32: the row's absmax; must be finite and >= 0
 *             (TRIT_E_SCALE otherwise; 0 is the scale of an all-zero row)
 *   w_scale   finite, > 0 (TRIT_E_SCALE)
 *   y_i32, y_f32, err_flag   as for trit_gemm
 */
TRIT_API trit_status trit_gemv(const uint8_t *planes, float w_scale, const int8_t *x_i8,
                               float x_scale, int64_t N, int64_t K, int32_t *y_i32,
                               float *y_f32, uint32_t *err_flag, trit_stream_t stream);

/*
 * Bits of trit_proj.flags and trit_qproj.flags (any other bit: TRIT_E_ARG).
 *
 * TRIT_PROJ_PLANES_READY: the entry's planes were complete before the kernel
 * that precedes this call on `stream` was launched (for instance packed, then
 * the stream synchronised), and nothing writes them while the call runs.  A
 * list whose every entry sets it may be launched with programmatic dependent
 * launch reading its planes into shared memory while the preceding kernel
 * still runs; the activations are read, and anything is written, only after
 * that kernel has completed.  Results are identical with or without the bit.
 */
#define TRIT_PROJ_PLANES_READY 1u

/* One product of a list: the arguments of trit_gemm, all device pointers. */
typedef struct trit_proj {
    const uint8_t *planes;
    const int8_t *x_i8;
    const float *x_scale;
    int32_t *y_i32;      /* may be NULL */
    float *y_f32;        /* may be NULL (not both) */
    int64_t M, N, K;
    float w_scale;
    uint32_t flags;      /* 0 or TRIT_PROJ_PLANES_READY */
} trit_proj;

/*
 * trit_gemm_many -- a list of independent products (e.g. the 210 ternary
 * projections of one decode token, "Tritium ..." -- Why it does not scale)
 * computed by one persistent launch per kernel kind, so that the cost of a
 * launch is paid once per list, not once per product.  `list` is a HOST array
 * of `count` entries (read before the call returns); entries must not write
 * overlapping outputs.  Results are those of calling trit_gemm on each entry.
 */
TRIT_API trit_status trit_gemm_many(const trit_proj *list, int32_t count, uint32_t *err_flag,
                                    trit_stream_t stream);

/* One fused decode product: an fp32 activation row quantised and multiplied in
 * the same launch.  M = 1. */
typedef struct trit_qproj {
    const uint8_t *planes;
    const float *x;      /* [K] fp32 activation row */
    int8_t *x_i8;        /* out, may be NULL: the row's codes, K_pad bytes, zero tail */
    float *x_scale;      /* out, may be NULL: the row's absmax */
    int32_t *y_i32;      /* may be NULL */
    float *y_f32;        /* may be NULL (not both) */
    int64_t N, K;
    float w_scale;
    uint32_t flags;      /* 0 or TRIT_PROJ_PLANES_READY */
} trit_qproj;

/*
 * trit_quant_gemv_many -- for each entry, trit_quant_act of its fp32 row
 * followed by trit_gemv, computed by one persistent launch for the whole list
 * (the quantiser runs inside the product kernel while it stages the
 * activations; no int8 round trip through memory).  Results -- y_i32, y_f32
 * and, when asked for, x_i8 and x_scale -- are bit-identical to the two-call
 * path.  K is limited to 73,728 (1,152 beats) per entry; longer rows return
 * TRIT_E_SHAPE and take the two-call path.  `list` is a host array.
 */
#define TRIT_MAX_FUSED_K 73728
TRIT_API trit_status trit_quant_gemv_many(const trit_qproj *list, int32_t count,
                                          uint32_t *err_flag, trit_stream_t stream);

/* One fused down projection of an IntMlp block ("Tritium: One Weight Format for
 * Ternary Inference ..." -- Numerics, IntMlp): the int32 gate and up outputs of
 * one token (a_gate, a_up, K values each, K = this projection's K) become this
 * projection's codes -- round-half-even(127 t / max|t|) of t = relu(a_gate)^2 *
 * a_up, exact -- and scale max|t| * S_g^2 * S_u (S = w * x_scale / 127), and
 * are multiplied, in the same launch.  M = 1. */
typedef struct trit_mlpproj {
    const uint8_t *planes;    /* the down projection, N x K */
    const int32_t *a_gate;    /* [K] gate output, device, 4-byte aligned */
    const int32_t *a_up;      /* [K] up output */
    const float *x_scale;     /* [1] the gate/up input's activation scale (device) */
    float w_gate, w_up;       /* the gate and up projections' weight scales */
    int8_t *h_i8;             /* out, may be NULL: the codes, K_pad bytes, zero tail */
    float *h_scale;           /* out, may be NULL: their scale */
    int32_t *y_i32;           /* may be NULL */
    float *y_f32;             /* may be NULL (not both) */
    int64_t N, K;
    float w_scale;            /* the down projection's */
    uint32_t reserved;        /* must be 0 */
} trit_mlpproj;

/*
 * trit_intmlp_gemv_many -- for each entry, trit_intmlp_quant of its gate and up
 * outputs followed by trit_gemv of the codes: y_i32, y_f32 and, when asked for,
 * h_i8 and h_scale are bit-identical to that two-call path.  Every CTA of the
 * launch forms the codes it needs while staging the row, so the int8 codes
 * make no round trip through memory; up to 8 entries share one launch (longer
 * lists take several).  K is limited to TRIT_MAX_FUSED_K (TRIT_E_SHAPE beyond);
 * w_gate, w_up and w_scale must be finite and > 0 (TRIT_E_SCALE).  `list` is a
 * host array; asynchronous on `stream`.
 */
TRIT_API trit_status trit_intmlp_gemv_many(const trit_mlpproj *list, int32_t count,
                                           uint32_t *err_flag, trit_stream_t stream);

/*
 * Batch-1 MLP blocks in two calls ("Tritium ..." -- Numerics, IntMlp):
 *   trit_mlp_gate_up: the fp32 row x (K values) quantised as trit_quant_act
 *     does (x_scale out) and multiplied by the gate and up planes (F x K each)
 *     into a_gate and a_up (int32, F values each); the maxima of
 *     |t| = |relu(a_gate)^2 * a_up| over each 32 columns and, per column, a
 *     signed fp32 form of t go to `tmax`.  One block per call is one launch
 *     whose CTAs form them from the rows they computed; lists whose rows do
 *     not fit one resident wave take the products on the streaming kernel and
 *     one more launch forming them.
 *   trit_mlp_down: the down projection (N x F) of the codes of t --
 *     round-half-even(127 t / max|t|), exact, max|t| reduced from `tmax` --
 *     with scale max|t| * S_g^2 * S_u (S = w * x_scale / 127): y_i32 / y_f32
 *     and, when asked for, h_i8 and h_scale.
 * Results are bit-identical to trit_quant_gemv_many([gate, up]) followed by
 * trit_intmlp_quant and trit_gemm of the down projection; a_gate, a_up and
 * x_scale are the first call's outputs.  trit_mlp_down reads what
 * trit_mlp_gate_up of the same blocks wrote: call it after that call on the
 * same stream, with x_scale, a_gate, a_up and tmax untouched in between.
 * Blocks whose rows exceed the pre-loading kernel's shared memory (K above
 * 13,312 or F above 8,960 columns) take the fused paths instead (tmax
 * unused), with the same results.  K and F are limited to TRIT_MAX_FUSED_K
 * (TRIT_E_SHAPE); w_gate, w_up and w_down must be finite and > 0
 * (TRIT_E_SCALE).
 *   x          [K] fp32, device, 4-byte aligned
 *   x_scale    [1] fp32 out
 *   a_gate, a_up  [F] int32 out, 16-byte aligned
 *   tmax       workspace of trit_mlp_tmax_bytes(F) bytes, 16-byte aligned
 *   h_i8       out, may be NULL: [F_pad] int8, zero tail, 16-byte aligned
 *   h_scale    out, may be NULL: [1] fp32
 *   y_i32, y_f32  [N] outputs, either may be NULL (not both)
 * `list` is a host array; up to 8 blocks share one launch of trit_mlp_down.
 */
typedef struct trit_mlp_block {
    const uint8_t *gate_planes;
    const uint8_t *up_planes;
    const uint8_t *down_planes;
    const float *x;
    float *x_scale;
    int32_t *a_gate;
    int32_t *a_up;
    void *tmax;
    int8_t *h_i8;
    float *h_scale;
    int32_t *y_i32;
    float *y_f32;
    int64_t K, F, N;
    float w_gate, w_up, w_down;
    uint32_t flags;           /* 0 or TRIT_PROJ_PLANES_READY (all three planes) */
} trit_mlp_block;

/* Bytes of the tmax workspace of a block with F gate/up rows (144 per 32 rows). */
TRIT_API int64_t trit_mlp_tmax_bytes(int64_t F);
TRIT_API trit_status trit_mlp_gate_up(const trit_mlp_block *list, int32_t count,
                                      uint32_t *err_flag, trit_stream_t stream);
TRIT_API trit_status trit_mlp_down(const trit_mlp_block *list, int32_t count,
                                   uint32_t *err_flag, trit_stream_t stream);

/*
 * trit_quant_act_folded -- quantise the normalised activations of a layer
 * without dividing by the rms ("Tritium ..." -- Numerics, Folded).  For each
 * row m of x (M x K fp32, row-major) and the norm gains g (K fp32):
 *   u = x (.) g (one fp32 rounding per element); x_i8 row m = the codes of u,
 *   exactly as trit_quant_act computes them (absmax codes are unchanged by the
 *   uniform factor 1/rms); x_scale[m] = max|u| / rms with
 *   rms = sqrt(sum(x^2) / K + eps) in double, rounded once to fp32 -- the
 *   absmax of the normalised row, so the products' dequantisation is that of
 *   the normalised activations.
 * eps >= 0 and finite (the pages give no value: it is the caller's).  A row
 * whose u holds a NaN or infinity gets codes 0, scale 0 and TRIT_ERR_NONFINITE.
 * x_i8 is M x K_pad with a zero tail, as trit_quant_act writes it.
 */
TRIT_API trit_status trit_quant_act_folded(const float *x, const float *gain, int64_t M, int64_t K,
                                           float eps, int8_t *x_i8, float *x_scale,
                                           uint32_t *err_flag, trit_stream_t stream);

/*
 * trit_intmlp_quant -- the squared-ReLU stage of the MLP, kept integer, fused
 * with the absmax quantisation of the next projection's input ("Tritium ..."
 * -- Numerics, IntMlp).  a_gate and a_up are the exact int32 outputs (M x N,
 * row-major, as trit_gemm writes y_i32) of the gate and up projections of the
 * same M input rows, whose scales are S_g = w_scale_gate * x_scale[m] / 127 and
 * S_u = w_scale_up * x_scale[m] / 127.  For each row:
 *   t_c = relu(a_gate_c)^2 * a_up_c, formed exactly (128-bit integers);
 *   h_i8 row m = round-half-even(127 * t_c / max|t|), an exact rational
 *   rounding (all 0 when max|t| = 0), zero tail to N_pad = 64 * ceil(N / 64);
 *   h_scale[m] = max|t| * (S_g^2 * S_u) in double, rounded once to fp32 (the
 *   absmax of relu(g)^2 u; max|t| enters as the double sum of its two 64-bit
 *   halves).
 * (h_i8, h_scale) are then the x_i8 / x_scale of the next projection (K' = N).
 * w_scale_* finite and > 0.  No data errors exist here.
 */
TRIT_API trit_status trit_intmlp_quant(const int32_t *a_gate, const int32_t *a_up, int64_t M,
                                       int64_t N, float w_scale_gate, float w_scale_up,
                                       const float *x_scale, int8_t *h_i8, float *h_scale,
                                       trit_stream_t stream);

/*
 * trit_gemm_noalloc -- trit_gemm with the same arguments, results and error
 * behaviour, that allocates no device memory in any form.  The methods on
 * ternary bit planes have nothing like it; it is a service for callers that
 * cannot let a library allocate while they run: engines that hand all device
 * memory to their own pools or caches up front and have no headroom left for
 * a driver allocation, and loops that must not meet an out-of-memory failure
 * or a memory-pool growth (which may wait on the device) in the middle of a
 * step.  trit_gemm's tensor-core path (M >= 13, K < 131072) needs a temporary
 * fp16 copy of the activations, which trit_gemm allocates on the stream; this
 * entry point puts that copy in one buffer of TRIT_NOALLOC_SCRATCH_BYTES that
 * is part of the library's device image instead.  The other paths use no
 * scratch and are those of trit_gemm.
 *
 *   Limit     the copy takes 2048 * ceil(M/16) * ceil(K/64) bytes when
 *             13 <= M <= 128 and K < 131072 (at most 32 MiB: always fits),
 *             32768 * ceil(M/256) * ceil(K/64) bytes when M > 128 and
 *             K < 131072, and 0 otherwise; the call returns TRIT_E_SCRATCH,
 *             enqueuing nothing, when that exceeds TRIT_NOALLOC_SCRATCH_BYTES
 *             (32 MiB: for M > 128, ceil(M/256) * ceil(K/64) <= 1024, e.g.
 *             M = 2048 with K <= 8192).  Split M to stay inside.
 *   Set-up    the first call on each device looks the buffer's address up with
 *             that device current (cudaGetSymbolAddress, which may load the
 *             library's device image and reserve the buffer) and keeps it for
 *             later calls.  Make that first call before any stream capture
 *             begins.  After cudaDeviceReset the kept address is stale: do not
 *             call this entry point again in that process.
 *   Zeroing   *err_flag must be zero before the call, as for trit_gemm.  The
 *             outputs and the buffer need not be: every byte of the buffer a
 *             call reads is written earlier in the same call.
 *   Overlap   there is one buffer per device.  Two calls on the same device
 *             whose work can run at the same time (different streams with no
 *             ordering between them, or host threads issuing to different
 *             streams) race on it and give wrong results.  Calls on one stream,
 *             or ordered by events, are safe; calls on different devices use
 *             different buffers.
 */
#define TRIT_NOALLOC_SCRATCH_BYTES (32ll * 1024 * 1024)
TRIT_API trit_status trit_gemm_noalloc(const uint8_t *planes, float w_scale, const int8_t *x_i8,
                                       const float *x_scale, int64_t M, int64_t N, int64_t K,
                                       int32_t *y_i32, float *y_f32, uint32_t *err_flag,
                                       trit_stream_t stream);

/* One quantisation of a list: the arguments of trit_quant_act. */
typedef struct trit_act {
    const float *x;
    int8_t *x_i8;
    float *x_scale;
    int64_t M, K;
} trit_act;

/* trit_quant_act_many -- a host list of independent quantisations, one launch. */
TRIT_API trit_status trit_quant_act_many(const trit_act *list, int32_t count,
                                         uint32_t *err_flag, trit_stream_t stream);

/* trit_read_probe -- measurement aid: read `bytes` (a multiple of 16, >= 16) of
 * the device buffer `buf` (16-byte aligned) once, with the 16-byte L1-bypassing
 * loads the products use for the planes, fully coalesced, and reduce them into
 * *sink (device u32, 4-byte aligned; its value is meaningless).  Timing this
 * launch gives the plain read rate of the device's memory, the reference the
 * products' HBM rate is compared with ("Tritium ..." -- Results: the weight
 * stream is the cost of a decode step).  Asynchronous on `stream`; TRIT_E_ARG
 * for null or misaligned pointers or a bad size. */
TRIT_API trit_status trit_read_probe(const void *buf, int64_t bytes, uint32_t *sink,
                                     trit_stream_t stream);

/* trit_issue_probe -- measurement aid: the per-SM completion rate of one
 * instruction that the select-accumulate kernels are built from (their decode
 * budget -- "Tritium ..." -- On popcount and The hardware core: the ternary
 * product is integer adds and bit logic, so these rates, not multiplies, bound
 * it).  Launches `blocks` CTAs of `threads` threads; every thread issues
 * 32 * iters instructions of kind `kind` in eight independent chains (64 * iters
 * for TRIT_PROBE_DP4A_LOP3, whose chains alternate the two).  Thread 0
 * of CTA i writes rec[3i] = its SM id, rec[3i+1] / rec[3i+2] = clock64() at
 * the start / end of the timed loop (after barriers).  Instructions per SM-clock
 * = (threads * 32 * iters * CTAs on that SM) / (latest end - earliest start on
 * that SM), all CTAs being resident at once (blocks <= SMs x CTAs per SM).
 * The shared-memory kinds read 4-byte words / 16-byte vectors at
 * conflict-free addresses (16 KB of static shared memory per CTA).
 *   kind     one of TRIT_PROBE_*
 *   blocks   >= 1;  threads: a multiple of 32 in [32, 512];  iters >= 1
 *   sink     device u32 (its value is meaningless);  rec: device u64 [3*blocks]
 * TRIT_E_ARG for a bad kind, size or pointer.  Asynchronous on `stream`. */
#define TRIT_PROBE_DP4A 0      /* dp4a.s32.s32 */
#define TRIT_PROBE_LOP3 1      /* lop3.b32 */
#define TRIT_PROBE_PRMT 2      /* prmt.b32 */
#define TRIT_PROBE_SHF 3       /* shf.l.wrap.b32 (funnel shift) */
#define TRIT_PROBE_IMAD 4      /* mad.lo.u32 */
#define TRIT_PROBE_IADD 5      /* add.u32 */
#define TRIT_PROBE_SHFL 6      /* shfl.sync.bfly.b32 */
#define TRIT_PROBE_LDS32 7     /* ld.shared.u32 (+ one xor) */
#define TRIT_PROBE_LDS128 8    /* ld.shared.v4.u32 (+ xors) */
#define TRIT_PROBE_DP4A_LOP3 9 /* dp4a then lop3 on each chain: both count */
#define TRIT_PROBE_DP4A_SU 10  /* dp4a.s32.u32 (signed by unsigned bytes) */
TRIT_API trit_status trit_issue_probe(int32_t kind, int32_t blocks, int32_t threads, int64_t iters,
                                      uint32_t *sink, uint64_t *rec, trit_stream_t stream);

/* trit_check_div127 -- diagnostic: every fp32 dequantisation divides by 127
 * ("Tritium: One Weight Format for Ternary Inference ..." -- Numerics: y_f32 =
 * ((y * w_scale) * x_scale) / 127, each step rounded once) with a multiply and
 * two FMAs (a reciprocal product and one Markstein residual correction) in place
 * of the IEEE divide.  This call evaluates both forms for all 2^32 float bit
 * patterns on the current device and stores the number of disagreements (NaN
 * against NaN counts as agreement) in *mismatches (host pointer; 0 means the two
 * are bit-identical).  Synchronous on the default stream; allocates 8 bytes of
 * device memory for the count.  TRIT_E_ARG for a null pointer; CUDA failures as
 * for the other calls (then *mismatches = UINT64_MAX). */
TRIT_API trit_status trit_check_div127(uint64_t *mismatches);

/*
 * ---- BITCOS weights -----------------------------------------------------------
 * "BITCOS: Intel's Ternary LLM Weight Format Goes Below 1.58 Bits" -- A bitmap
 * and a sign; Decoding is the other half of the bill.  A ternary matrix as a
 * presence bitmap (one bit per weight, set for a non-zero weight) and a sign
 * vector (one bit per non-zero weight in the same order, set for -1): 2 - z
 * bits per weight at zero density z, against 2 for the planes.  Here in a
 * blocked form so that every row can be started on its own:
 *   bitmap   uint64 [N][ceil(K/64)]: bit c%64 of word [r][c/64] = (W[r][c] != 0);
 *            bits past K are 0;
 *   sign_off uint32 [N+1]: sign_off[0] = 0, sign_off[r+1] = sign_off[r] +
 *            ceil(nnz_r / 32) (nnz_r: row r's non-zeros);
 *   signs    uint32 [sign_off[N] + 2]: the k-th non-zero of row r (column order)
 *            is -1 when bit k%32 of word sign_off[r] + k/32 is set; all other
 *            bits, and the last two words, are 0.
 * Row r's sign bits, in order and cut to nnz_r, are row r's part of the page's
 * flat sign vector; its bitmap bits are row r's part of the flat bitmap.
 */
#define TRIT_BITCOS_MAX_K 16384

/* trit_bitcos_pack -- HOST code, no CUDA call: W [N][K] int8 in {-1, 0, +1}
 * (host memory, row-major, K columns, no padding) -> the three arrays above, in
 * host memory.  Call with signs == NULL first: *sign_words receives the length of
 * `signs` (sign_off[N] + 2) and bitmap / sign_off may be NULL.  Then call with
 * bitmap [N * ceil(K/64)], sign_off [N+1] and signs [*sign_words].
 *   TRIT_E_ARG    w or sign_words NULL; signs given without bitmap or sign_off
 *   TRIT_E_SHAPE  N or K outside [1, 2^31) x [1, TRIT_BITCOS_MAX_K], or more
 *                 than 2^32 - 3 sign words
 *   TRIT_E_VALUE  a weight outside {-1, 0, +1} (the outputs are then undefined)
 */
TRIT_API trit_status trit_bitcos_pack(const int8_t *w, int64_t N, int64_t K, uint64_t *bitmap,
                                      uint32_t *sign_off, uint32_t *signs, int64_t *sign_words);

/* One product of trit_bitcos_gemv_many: y = W x for ONE activation row.
 * All pointers are device pointers. */
typedef struct trit_bitcos_proj {
    const uint64_t *bitmap;     /* [N][ceil(K/64)], 16-byte aligned */
    const uint32_t *sign_off;   /* [N+1], 4-byte aligned */
    const uint32_t *signs;      /* [sign_words], 4-byte aligned */
    const int8_t *x_i8;         /* [K_pad] activation codes, 16-byte aligned (columns >= K ignored) */
    const float *x_scale;       /* [1] */
    int32_t *y_i32;             /* [N], or NULL */
    float *y_f32;               /* [N], or NULL (not both) */
    int64_t N, K;
    int64_t sign_words;         /* length of `signs`; reads are clamped to it */
    float w_scale;              /* finite, > 0 */
    int32_t reserved;           /* must be 0 */
} trit_bitcos_proj;

/* trit_bitcos_gemv_many -- y = W x for every product of the host list, W in the
 * BITCOS form above: exact int32 sums, y_f32 = (((float)y * w_scale) *
 * x_scale) / 127 as for trit_gemm, identical bits to trit_gemm on the planes of
 * the same W.  A list longer than TRIT_MAX_LIST_PER_LAUNCH is split.  The first
 * call on each device uploads a 64 KB table (cudaMemcpyToSymbol, synchronous):
 * make it before any stream capture.  The arrays must be those trit_bitcos_pack
 * produced (inconsistent ones give wrong results; every read stays inside the
 * arrays' stated lengths).  TRIT_E_ARG / TRIT_E_SHAPE / TRIT_E_SCALE as for
 * trit_gemm_many (K <= TRIT_BITCOS_MAX_K). */
TRIT_API trit_status trit_bitcos_gemv_many(const trit_bitcos_proj *list, int32_t count,
                                           trit_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TRIT_H */

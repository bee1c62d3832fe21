/*
 * trit_oracle.c -- reference CPU implementation of the ternary bit-plane
 * select-accumulate path.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
 * CPU-baseline leg call this code; the product library never does, and this
 * file shares no code, header, table or constant with it.
 *
 * It is deliberately plain and slow: every weight is decoded bit by bit into
 * one int8, products are accumulated in int64, and nothing is blocked, fused,
 * vectorised or reordered.  Single-threaded.
 *
 * Sources (page title -- section):
 *   [FMT] "The .trit format, version 1" -- 2.3 Ternary payload; 4 Validation
 *   [TRI] "Tritium: One Weight Format for Ternary Inference on Commodity CPUs
 *          and Multiplier-Free Hardware" -- The .trit v1 layout; Invariants;
 *          On popcount; The hardware core; Numerics; Why exactness, concretely
 *   [BITCOS] "BITCOS: Intel's Ternary LLM Weight Format Goes Below 1.58 Bits"
 *          -- A bitmap and a sign
 *
 * Readings where the pages are silent (the activation quantiser formula, the
 * zero row, the dequantisation order) are stated at each function.
 *
 * Return codes are bit masks:
 *   1  both planes set in one weight position (P1)
 *   2  padding bit set past the last column (P2)
 *   4  value outside {-1, 0, +1} handed to the packer
 *   8  non-finite activation handed to the quantiser
 *   32 accumulator outside the int32 range
 *   64 bad argument
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define OR_P1          1
#define OR_P2          2
#define OR_NOT_TERNARY 4
#define OR_NONFINITE   8
#define OR_OVERFLOW    32
#define OR_ARG         64

/* [FMT] 2.3: beats_per_row = ceil(cols / 64). */
int64_t oracle_beats_per_row(int64_t cols) { return (cols + 63) / 64; }

/* [FMT] 2.3: byte_len = rows * beats_per_row * 16. */
int64_t oracle_payload_bytes(int64_t rows, int64_t cols)
{
    return rows * oracle_beats_per_row(cols) * 16;
}

/* [FMT] 2.3: beat b of row r is the 16 bytes at (r * beats_per_row + b) * 16. */
static const uint8_t *beat_at(const uint8_t *payload, int64_t cols, int64_t r, int64_t b)
{
    return payload + (r * oracle_beats_per_row(cols) + b) * 16;
}

/* [FMT] 2.3: bytes 0..8 hold pos, bytes 8..16 hold neg, each a little-endian
 * u64 whose bit k is the k-th least significant bit.  Bit k of a little-endian
 * u64 is bit (k % 8) of byte (k / 8). */
static int pos_bit(const uint8_t *beat, int k) { return (beat[k / 8] >> (k % 8)) & 1; }
static int neg_bit(const uint8_t *beat, int k) { return (beat[8 + k / 8] >> (k % 8)) & 1; }

/*
 * Pack an int8 ternary matrix (rows x cols, row-major) into the .trit v1
 * ternary payload.  [FMT] 2.3: bit k of pos set <=> W[r][b*64+k] = +1, bit k
 * of neg set <=> W[r][b*64+k] = -1, neither set <=> 0; padding bits past cols
 * stay clear (P2).  A value outside {-1, 0, +1} is rejected, with its linear
 * index in *bad.
 */
int oracle_pack(const int8_t *w, int64_t rows, int64_t cols, uint8_t *payload, int64_t *bad)
{
    if (rows < 0 || cols < 0) return OR_ARG;
    memset(payload, 0, (size_t)oracle_payload_bytes(rows, cols));
    int64_t bpr = oracle_beats_per_row(cols);
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t c = 0; c < cols; c++) {
            int8_t v = w[r * cols + c];
            int64_t b = c / 64;
            int k = (int)(c % 64);
            uint8_t *beat = payload + (r * bpr + b) * 16;
            if (v == 1) {
                beat[k / 8] |= (uint8_t)(1u << (k % 8));
            } else if (v == -1) {
                beat[8 + k / 8] |= (uint8_t)(1u << (k % 8));
            } else if (v != 0) {
                if (bad) *bad = r * cols + c;
                return OR_NOT_TERNARY;
            }
        }
    }
    return 0;
}

/*
 * Check both payload invariants.  [TRI] Invariants / [FMT] 2.3:
 *   P1: pos AND neg = 0 in every beat, padding included;
 *   P2: on every row's last beat, (pos OR neg) AND NOT tail = 0, where tail is
 *       all ones when cols % 64 = 0 and (1 << (cols % 64)) - 1 otherwise, the
 *       shift done in 64 bits.
 * Written here bit by bit: a padding bit is one whose column b*64+k >= cols.
 * Returns the OR of the kinds found (0 = clean) and, in *first, the smallest
 * offending bit position (r * beats_per_row + b) * 64 + k over both kinds.
 */
int oracle_verify(const uint8_t *payload, int64_t rows, int64_t cols, int64_t *first)
{
    int64_t bpr = oracle_beats_per_row(cols);
    int kinds = 0;
    int64_t best = -1;
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < bpr; b++) {
            const uint8_t *beat = beat_at(payload, cols, r, b);
            for (int k = 0; k < 64; k++) {
                int p = pos_bit(beat, k), n = neg_bit(beat, k);
                int here = 0;
                if (p && n) here |= OR_P1;
                if ((p || n) && b * 64 + k >= cols) here |= OR_P2;
                if (here) {
                    kinds |= here;
                    if (best < 0) best = (r * bpr + b) * 64 + k;
                }
            }
        }
    }
    if (first) *first = best;
    return kinds;
}

/*
 * Inverse of oracle_pack.  A weight position with both bits set is rejected
 * ([FMT] 2.3, P1: every consumer must treat it as an error), with its bit
 * position (as in oracle_verify) in *bad.  Padding bits are not columns and
 * are not read.
 */
int oracle_unpack(const uint8_t *payload, int64_t rows, int64_t cols, int8_t *w, int64_t *bad)
{
    int64_t bpr = oracle_beats_per_row(cols);
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < bpr; b++) {
            const uint8_t *beat = beat_at(payload, cols, r, b);
            for (int k = 0; k < 64; k++) {
                int p = pos_bit(beat, k), n = neg_bit(beat, k);
                if (p && n) {
                    if (bad) *bad = (r * bpr + b) * 64 + k;
                    return OR_P1;
                }
                int64_t c = b * 64 + k;
                if (c < cols) w[r * cols + c] = (int8_t)(p ? 1 : (n ? -1 : 0));
            }
        }
    }
    return 0;
}

/*
 * Per-token absmax activation quantiser.  [TRI] Numerics names the recipe
 * (per-token absmax int8, codes invariant under a uniform positive scale) but
 * prints no formula; the reading used here, for each row of x (M x K, fp32):
 *   a     = max_c |x_c|                      (exact in fp32)
 *   inv   = 127.0f / a                       (IEEE fp32 division)
 *   q_c   = clamp(rint(x_c * inv), -127, 127) (fp32 product, ties to even)
 *   scale = a
 * Special cases:
 *   - any non-finite x_c: the row is rejected (row_err = 8), q = 0, scale = 0;
 *   - a = 0: q = 0 and scale = 0;
 *   - a < 2^-96, where 127/a could overflow: x and a are first multiplied by
 *     2^96, which is exact, so the codes are those of the row scaled into the
 *     normal range (the uniform-scale invariance above).
 * q is written with row stride ldq >= K; columns K..ldq-1 are zero
 * ([FMT] 2.3: activation buffers are sized beats_per_row * 64 with a zero tail).
 * Returns the OR of the row errors.
 */
int oracle_quant(const float *x, int64_t M, int64_t K, int64_t ldq, int8_t *q, float *scale,
                 uint8_t *row_err)
{
    int any = 0;
    for (int64_t m = 0; m < M; m++) {
        const float *xr = x + m * K;
        int8_t *qr = q + m * ldq;
        memset(qr, 0, (size_t)ldq);
        row_err[m] = 0;
        scale[m] = 0.0f;
        int finite = 1;
        float a = 0.0f;
        for (int64_t c = 0; c < K; c++) {
            if (!isfinite(xr[c])) finite = 0;
            else if (fabsf(xr[c]) > a) a = fabsf(xr[c]);
        }
        if (!finite) {
            row_err[m] = OR_NONFINITE;
            any |= OR_NONFINITE;
            continue;
        }
        if (a == 0.0f) continue;
        float pre = 1.0f;
        if (a < 0x1p-96f) pre = 0x1p96f;
        float inv = 127.0f / (a * pre);
        for (int64_t c = 0; c < K; c++) {
            float v = rintf((xr[c] * pre) * inv);
            if (v > 127.0f) v = 127.0f;
            if (v < -127.0f) v = -127.0f;
            qr[c] = (int8_t)v;
        }
        scale[m] = a;
    }
    return any;
}

/*
 * Decode one payload row to one int8 per column, bit by bit ([TRI]
 * Verification: the oracle expands bit planes to one i8 per weight).  Every
 * bit of every beat of the row, padding included, is checked for P1.
 * Returns 0 or OR_P1 with the first offending bit position in *bad.
 */
static int decode_row(const uint8_t *payload, int64_t cols, int64_t r, int8_t *wrow, int64_t *bad)
{
    int64_t bpr = oracle_beats_per_row(cols);
    for (int64_t b = 0; b < bpr; b++) {
        const uint8_t *beat = beat_at(payload, cols, r, b);
        for (int k = 0; k < 64; k++) {
            int p = pos_bit(beat, k), n = neg_bit(beat, k);
            if (p && n) {
                if (bad) *bad = (r * bpr + b) * 64 + k;
                return OR_P1;
            }
            int64_t c = b * 64 + k;
            if (c < cols) wrow[c] = (int8_t)(p ? 1 : (n ? -1 : 0));
        }
    }
    return 0;
}

/*
 * y = W x for the selected payload rows, plus its fp32 dequantisation.
 *   payload : rows N x cols K as in [FMT] 2.3
 *   x       : M activation rows of int8 with row stride ldx (>= K); only
 *             columns < K are read -- padding columns do not exist
 *   x_scale : M per-row scales (the absmax of each quantised row)
 *   sel     : indices of the payload rows to evaluate (NULL = all N, in order)
 *   y_i32, y_f32 : M x nsel, row-major
 * For each selected row the weights are decoded to int8 and
 *   acc = sum_c W[r][c] * x[m][c]   in int64,
 * which must lie in the int32 range ([TRI] The hardware core: a 32-bit
 * accumulator, with -128 activations widened before they are negated).
 * Dequantisation, in the order the configuration states it, one fp32
 * round-to-nearest step at a time, without contraction ([TRI] Why exactness:
 * scale by each factor in turn):
 *   y_f32 = (((float)acc * w_scale) * x_scale[m]) / 127.0f
 * A row containing a both-bits-set position is rejected (row_err = 1, its
 * outputs 0); the return value is the OR of the row errors.
 */
int oracle_gemm(const uint8_t *payload, float w_scale, const int8_t *x, int64_t ldx,
                const float *x_scale, int64_t M, int64_t N, int64_t K, const int64_t *sel,
                int64_t nsel, int32_t *y_i32, float *y_f32, uint8_t *row_err, int8_t *scratch)
{
    int any = 0;
    if (sel == NULL) nsel = N;
    for (int64_t i = 0; i < nsel; i++) {
        int64_t r = sel ? sel[i] : i;
        if (r < 0 || r >= N) return OR_ARG;
        row_err[i] = (uint8_t)decode_row(payload, K, r, scratch, NULL);
        for (int64_t m = 0; m < M; m++) {
            y_i32[m * nsel + i] = 0;
            y_f32[m * nsel + i] = 0.0f;
        }
        if (row_err[i]) {
            any |= row_err[i];
            continue;
        }
        for (int64_t m = 0; m < M; m++) {
            const int8_t *xr = x + m * ldx;
            int64_t acc = 0;
            for (int64_t c = 0; c < K; c++) acc += (int64_t)scratch[c] * (int64_t)xr[c];
            if (acc > INT32_MAX || acc < INT32_MIN) {
                row_err[i] |= OR_OVERFLOW;
                any |= OR_OVERFLOW;
                continue;
            }
            float f = (float)(int32_t)acc;
            f = f * w_scale;
            f = f * x_scale[m];
            f = f / 127.0f;
            y_i32[m * nsel + i] = (int32_t)acc;
            y_f32[m * nsel + i] = f;
        }
    }
    return any;
}

/*
 * The bit-serial popcount formulation ([TRI] On popcount), kept as a second,
 * independent evaluation of the integer result.  Writing each int8 activation
 * in two's complement, x = -128*b7 + sum_{j<7} 2^j * b_j, gives
 *   y = sum_{j<7} 2^j (popc(pos & X_j) - popc(neg & X_j))
 *       - 128 (popc(pos & X_7) - popc(neg & X_7))
 * where X_j is the 64-bit mask of bit j of the activations of one beat.  The
 * masks are built per beat with columns >= K cleared.  Only the int32 result
 * is produced; a both-bits-set position makes the row's result unspecified
 * here (oracle_gemm is the one that rejects).
 */
static int popcount64(uint64_t v)
{
    int n = 0;
    while (v) {
        n += (int)(v & 1u);
        v >>= 1;
    }
    return n;
}

int oracle_gemm_popcount(const uint8_t *payload, const int8_t *x, int64_t ldx, int64_t M,
                         int64_t N, int64_t K, int32_t *y_i32)
{
    int64_t bpr = oracle_beats_per_row(K);
    for (int64_t r = 0; r < N; r++) {
        for (int64_t m = 0; m < M; m++) {
            const int8_t *xr = x + m * ldx;
            int64_t acc = 0;
            for (int64_t b = 0; b < bpr; b++) {
                const uint8_t *beat = beat_at(payload, K, r, b);
                uint64_t pos = 0, neg = 0;
                for (int i = 0; i < 8; i++) {
                    pos |= (uint64_t)beat[i] << (8 * i);
                    neg |= (uint64_t)beat[8 + i] << (8 * i);
                }
                for (int j = 0; j < 8; j++) {
                    uint64_t xj = 0;
                    for (int k = 0; k < 64; k++) {
                        int64_t c = b * 64 + k;
                        if (c < K && (((uint8_t)xr[c] >> j) & 1u)) xj |= (uint64_t)1 << k;
                    }
                    int64_t d = (int64_t)popcount64(pos & xj) - (int64_t)popcount64(neg & xj);
                    acc += (j == 7) ? -128 * d : ((int64_t)1 << j) * d;
                }
            }
            if (acc > INT32_MAX || acc < INT32_MIN) return OR_OVERFLOW;
            y_i32[m * N + r] = (int32_t)acc;
        }
    }
    return 0;
}

/*
 * [TRI] Numerics -- Folded.  The 1/rms of the normalisation never touches the
 * elements: absmax codes are unchanged by a uniform positive scale, so they are
 * the codes of u = x (.) g (the elements times the norm gains, each product one
 * fp32 rounding), computed exactly as oracle_quant computes them, and the rms
 * appears only in the row's scale.  Readings (the pages give neither the rms
 * formula nor its epsilon): rms = sqrt(sum over c of x_c^2 / K + eps) in
 * double, summed in column order; the scale is (float)(a / rms) with a = max|u|,
 * i.e. the absmax of the normalised row.  A row with a non-finite x, g or u is
 * rejected as in oracle_quant (codes 0, scale 0, row error 8).
 */
int oracle_quant_folded(const float *x, const float *g, int64_t M, int64_t K, double eps,
                        int64_t ldq, int8_t *q, float *scale, uint8_t *row_err, float *u)
{
    int any = 0;
    for (int64_t m = 0; m < M; m++) {
        const float *xr = x + m * K;
        double s2 = 0.0;
        for (int64_t c = 0; c < K; c++) {
            u[c] = xr[c] * g[c];
            s2 += (double)xr[c] * (double)xr[c];
        }
        any |= oracle_quant(u, 1, K, ldq, q + m * ldq, scale + m, row_err + m);
        if (row_err[m] == 0 && scale[m] != 0.0f) {
            const double rms = sqrt(s2 / (double)K + eps);
            scale[m] = (float)((double)scale[m] / rms);
        }
    }
    return any;
}

/*
 * [TRI] Numerics -- IntMlp.  With the gate output g = a_g S_g and the up output
 * u = a_u S_u (integer products times uniform positive scales), the squared-ReLU
 * product relu(g)^2 u equals t K with the integer t = relu(a_g)^2 a_u and
 * K = S_g^2 S_u; it never exists in floating point.  The next projection's
 * activations h = t K are quantised per row by absmax, and since K > 0 is
 * uniform the codes are those of t.  Readings:
 *   - t is formed in 128-bit integers (exact for any int32 inputs; the page
 *     bounds it below 2^55 for its model, where it equals the i64 value);
 *   - codes q_c = round-half-even(127 t_c / A) with A = max_c |t_c|, an exact
 *     rational rounding (|q_c| <= 127 without a clamp); all 0 when A = 0;
 *   - the row's scale is the absmax of h, A K, in double:
 *     S_g = w_g * s / 127, S_u = w_u * s / 127 (s the input row's x_scale),
 *     K = (S_g * S_g) * S_u, A as a double = hi * 2^64 + lo (its two 64-bit
 *     halves, each converted, then summed), scale = (float)(A * K).
 * ag, au: M rows of N int32 with row stride ld; q: M rows of ldq >= N codes,
 * zero past N.
 */
typedef __int128 i128;

static i128 intmlp_t(int32_t g, int32_t u)
{
    if (g <= 0) return 0;
    return (i128)g * (i128)g * (i128)u;
}

static int round_ratio_127(i128 t, i128 A)
{
    const int neg = t < 0;
    const i128 n = 127 * (neg ? -t : t);
    i128 q = n / A;
    const i128 r = n - q * A;
    if (2 * r > A || (2 * r == A && (q & 1))) q += 1;
    return (int)(neg ? -q : q);
}

int oracle_intmlp_quant(const int32_t *ag, const int32_t *au, int64_t M, int64_t N, int64_t ld,
                        float w_g, float w_u, const float *x_scale, int64_t ldq, int8_t *q,
                        float *h_scale)
{
    for (int64_t m = 0; m < M; m++) {
        i128 A = 0;
        for (int64_t c = 0; c < N; c++) {
            i128 t = intmlp_t(ag[m * ld + c], au[m * ld + c]);
            if (t < 0) t = -t;
            if (t > A) A = t;
        }
        int8_t *qr = q + m * ldq;
        memset(qr, 0, (size_t)ldq);
        for (int64_t c = 0; c < N && A > 0; c++)
            qr[c] = (int8_t)round_ratio_127(intmlp_t(ag[m * ld + c], au[m * ld + c]), A);
        const double sg = (double)w_g * (double)x_scale[m] / 127.0;
        const double su = (double)w_u * (double)x_scale[m] / 127.0;
        const double k = (sg * sg) * su;
        const uint64_t hi = (uint64_t)(A >> 64), lo = (uint64_t)A;
        const double a = (double)hi * 18446744073709551616.0 + (double)lo;
        h_scale[m] = (float)(a * k);
    }
    return 0;
}

/*
 * BITCOS ([BITCOS] "BITCOS: Intel's Ternary LLM Weight Format Goes Below 1.58
 * Bits" -- A bitmap and a sign).  Two arrays: a presence bitmap with one bit
 * per weight (set when the weight is non-zero) and a sign vector with one bit
 * per non-zero weight, in the same order (set when the weight is -1).  Bits
 * are filled from the least significant bit of each byte upward, as the
 * page's packer does.  Rate: n + nnz bits, i.e. 2 - z bits per weight at zero
 * density z.
 *
 * oracle_bitcos_pack_flat: q[0..n) in {-1, 0, +1} -> bitmap[ceil(n/8)],
 * signs[ceil(nnz/8)] (the caller sizes signs for n weights), *nnz.  Returns
 * OR_NOT_TERNARY (nothing defined) for a value outside {-1, 0, +1}.
 */
int oracle_bitcos_pack_flat(const int8_t *q, int64_t n, uint8_t *bitmap, uint8_t *signs,
                            int64_t *nnz)
{
    if (n < 0) return OR_ARG;
    for (int64_t i = 0; i < n; i++)
        if (q[i] < -1 || q[i] > 1) return OR_NOT_TERNARY;
    memset(bitmap, 0, (size_t)((n + 7) / 8));
    memset(signs, 0, (size_t)((n + 7) / 8));
    int64_t k = 0;
    for (int64_t i = 0; i < n; i++) {
        if (q[i] == 0) continue;
        bitmap[i / 8] |= (uint8_t)(1u << (i % 8));
        if (q[i] < 0) signs[k / 8] |= (uint8_t)(1u << (k % 8));
        k++;
    }
    *nnz = k;
    return 0;
}

/* The inverse: walk the bitmap; each set bit takes the next sign bit. */
int oracle_bitcos_unpack_flat(const uint8_t *bitmap, const uint8_t *signs, int64_t n, int8_t *q)
{
    int64_t k = 0;
    for (int64_t i = 0; i < n; i++) {
        if ((bitmap[i / 8] >> (i % 8)) & 1) {
            q[i] = ((signs[k / 8] >> (k % 8)) & 1) ? (int8_t)-1 : (int8_t)1;
            k++;
        } else {
            q[i] = 0;
        }
    }
    return 0;
}

/*
 * The blocked form of the same two arrays for a matrix of `rows` x `cols`
 * weights, so that a kernel can start any row (the page: a production kernel
 * aligns both arrays to its block size).  Reading: the block is one row --
 *   bitmap  uint64 [rows][B], B = ceil(cols/64): bit c%64 of word [r][c/64] is
 *           row r's presence bit of column c; bits past cols are 0;
 *   sign_off uint32 [rows+1]: sign_off[0] = 0, sign_off[r+1] = sign_off[r] +
 *           ceil(nnz_r / 32);
 *   signs   uint32 [sign_off[rows] + 2]: the k-th non-zero of row r (column
 *           order) has its sign at bit k%32 of word sign_off[r] + k/32; every
 *           other bit is 0, and so are the last two words.
 * Row r's sign bits, taken in order and cut to nnz_r, are row r's part of the
 * flat sign vector.  oracle_bitcos_blocked_words gives sign_off[rows] (call it
 * first to size signs); oracle_bitcos_pack_blocked fills the three arrays.
 */
int64_t oracle_bitcos_blocked_words(const int8_t *w, int64_t rows, int64_t cols)
{
    int64_t words = 0;
    for (int64_t r = 0; r < rows; r++) {
        int64_t nnz = 0;
        for (int64_t c = 0; c < cols; c++) nnz += w[r * cols + c] != 0;
        words += (nnz + 31) / 32;
    }
    return words;
}

int oracle_bitcos_pack_blocked(const int8_t *w, int64_t rows, int64_t cols, uint64_t *bitmap,
                               uint32_t *sign_off, uint32_t *signs)
{
    const int64_t B = (cols + 63) / 64;
    if (rows < 0 || cols < 0) return OR_ARG;
    for (int64_t i = 0; i < rows * cols; i++)
        if (w[i] < -1 || w[i] > 1) return OR_NOT_TERNARY;
    memset(bitmap, 0, (size_t)(rows * B) * sizeof(uint64_t));
    int64_t off = 0;
    sign_off[0] = 0;
    for (int64_t r = 0; r < rows; r++) {
        int64_t k = 0;
        for (int64_t c = 0; c < cols; c++) {
            const int8_t v = w[r * cols + c];
            if (v == 0) continue;
            bitmap[r * B + c / 64] |= (uint64_t)1 << (c % 64);
            if (k % 32 == 0) signs[off + k / 32] = 0;
            if (v < 0) signs[off + k / 32] |= (uint32_t)1 << (k % 32);
            k++;
        }
        off += (k + 31) / 32;
        sign_off[r + 1] = (uint32_t)off;
    }
    signs[off] = 0;
    signs[off + 1] = 0;
    return 0;
}

/*
 * y = W x for one activation row with W given in the blocked BITCOS form:
 * each row is decoded by walking its bitmap and taking the next sign bit at
 * every set bit, then accumulated in int64 against x (int8, columns < cols),
 * and dequantised exactly as oracle_gemm does:
 *   y_f32 = (((float)acc * w_scale) * x_scale) / 127.0f
 * `sel` selects rows (NULL: all).  Returns OR_OVERFLOW if an accumulator
 * leaves the int32 range (that row's outputs are 0).
 */
int oracle_bitcos_gemv(const uint64_t *bitmap, const uint32_t *sign_off, const uint32_t *signs,
                       int64_t rows, int64_t cols, float w_scale, const int8_t *x, float x_scale,
                       const int64_t *sel, int64_t nsel, int32_t *y_i32, float *y_f32)
{
    const int64_t B = (cols + 63) / 64;
    int any = 0;
    if (sel == NULL) nsel = rows;
    for (int64_t i = 0; i < nsel; i++) {
        const int64_t r = sel ? sel[i] : i;
        if (r < 0 || r >= rows) return OR_ARG;
        int64_t acc = 0, k = 0;
        for (int64_t c = 0; c < cols; c++) {
            if (!((bitmap[r * B + c / 64] >> (c % 64)) & 1)) continue;
            const int64_t word = (int64_t)sign_off[r] + k / 32;
            const int neg = (signs[word] >> (k % 32)) & 1;
            acc += neg ? -(int64_t)x[c] : (int64_t)x[c];
            k++;
        }
        y_i32[i] = 0;
        y_f32[i] = 0.0f;
        if (acc > INT32_MAX || acc < INT32_MIN) {
            any |= OR_OVERFLOW;
            continue;
        }
        float f = (float)(int32_t)acc;
        f = f * w_scale;
        f = f * x_scale;
        f = f / 127.0f;
        y_i32[i] = (int32_t)acc;
        y_f32[i] = f;
    }
    return any;
}

// Internal declarations shared by the libtrit translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "trit.h"

namespace trit {

// ---- sizes -----------------------------------------------------------------

constexpr int64_t kMaxK = (int64_t(1) << 24) - 1;     // 128*K < 2^31
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;

__host__ __device__ inline int64_t beats_per_row(int64_t K) { return (K + 63) / 64; }

// ---- device helpers ---------------------------------------------------------

// d = c + sum_i a.s8[i] * b.u8[i]: signed activation bytes against unsigned
// mask bytes (mask bytes hold 0 or 2^j, up to 128).
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// d = c + sum_i a.s8[i] * b.s8[i].
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// Byte permute: result byte i is byte sel.nibble[i] of {b:a} (8 bytes); a
// nibble with bit 3 set replicates the sign bit of the selected byte.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// 16-byte streaming load of read-once data: not kept in L1.  TRIT_LDG_L2_FETCH
// selects the L2 fetch granularity hint on a miss (0: default, 128 or 256 bytes).
#ifndef TRIT_LDG_L2_FETCH
#define TRIT_LDG_L2_FETCH 0
#endif
__device__ __forceinline__ uint4 ldg_stream(const uint4 *p) {
    uint4 v;
#if TRIT_LDG_L2_FETCH == 256
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#elif TRIT_LDG_L2_FETCH == 128
    asm volatile("ld.global.nc.L1::no_allocate.L2::128B.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#else
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
#endif
    return v;
}

// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned source) into L2;
// no registers are held and nothing waits for it.
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// f / 127 rounded to nearest even -- the result of one IEEE division -- at the
// cost of a multiply and two FMAs: q = RN(f * c) with c = RN(1/127), then one
// correction step in the manner of Markstein (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): the residual r = f - 127 q is exact under an FMA, and
// q + r c is rounded once.  Zeros, non-finite values and magnitudes outside
// [2^-100, 2^120] take the IEEE divide.  Over the fast range the result equals
// __fdiv_rn(f, 127.0f) for every float: trit_check_div127 compares all 2^32
// bit patterns on the device.
__device__ __forceinline__ float div127_rn(float f) {
    const float a = fabsf(f);
    if (!(a >= 0x1p-100f && a <= 0x1p120f)) return __fdiv_rn(f, 127.0f);
    const float c = 0x1.020408p-7f;   // RN(1/127)
    const float q = __fmul_rn(f, c);
    const float r = __fmaf_rn(-q, 127.0f, f);
    return __fmaf_rn(r, c, q);
}

// ---- IntMlp arithmetic ("Tritium: One Weight Format for Ternary Inference ..." --
// Numerics, IntMlp): t = relu(a_g)^2 * a_u kept integer; the next projection's
// codes are round-half-even(127 t / max|t|) and its scale is max|t| * S_g^2 S_u
// with S = w_scale * x_scale / 127.  Shared by the standalone quantiser and the
// down-projection staging so both give the same codes and scale.

typedef unsigned __int128 trit_u128;

// |t| (exact, < 2^93) and the sign of t.
__device__ __forceinline__ trit_u128 intmlp_abs_t(int32_t ag, int32_t au, bool &neg) {
    neg = false;
    if (ag <= 0 || au == 0) return 0;
    const uint64_t g2 = uint64_t(ag) * uint64_t(ag);                  // < 2^62
    neg = au < 0;
    const uint64_t uu = neg ? uint64_t(-int64_t(au)) : uint64_t(au);   // <= 2^31
    return trit_u128(g2) * trit_u128(uu);
}

// Per-row constants of the code computation: A = max|t| (hi:lo), whether the
// 64-bit path applies (A < 2^56, so 127 A < 2^63) and k = 127 / A in fp32.
struct IntMlpRow {
    trit_u128 A;
    bool small, zero;
    float k;    // 127 / A in fp32 when A < 2^56 (the 64-bit path), else 0
    float kf;   // 127 / fl(A) in fp32 for any A > 0 (the estimate of intmlp_code_est)
};
__device__ __forceinline__ IntMlpRow intmlp_row(uint64_t hi, uint64_t lo) {
    IntMlpRow R;
    R.A = (trit_u128(hi) << 64) | trit_u128(lo);
    R.zero = hi == 0 && lo == 0;
    R.small = hi == 0 && lo < (uint64_t(1) << 56);
    R.k = R.small && !R.zero ? __fdiv_rn(127.0f, __ull2float_rn(lo)) : 0.0f;
    const float af = __fadd_rn(__fmul_rn(__ull2float_rn(hi), 0x1p64f), __ull2float_rn(lo));
    R.kf = R.zero ? 0.0f : __fdiv_rn(127.0f, af);
    return R;
}

// round-half-even(127 a / A) for 0 <= a <= A, A > 0 (the quotient is <= 127).
// A < 2^56: q0 = trunc(fl(a) * k) is within one of floor(127 a / A) (fp32
// relative error below 2^-21, times at most 127), then the exact remainder
// r = 127 a - q A in 64-bit integers fixes q to the floor and decides the
// rounding.  Otherwise: a 7-step binary search in 128-bit integers.
__device__ __forceinline__ int round_127_ratio_small(uint64_t a64, uint64_t A, float k) {
    int q = __float2int_rz(__fmul_rn(__ull2float_rn(a64), k));
    q = q > 127 ? 127 : q;
    int64_t r = int64_t(a64 * 127u) - int64_t(q) * int64_t(A);
    if (r < 0) {
        --q;
        r += int64_t(A);
    } else if (r >= int64_t(A)) {
        ++q;
        r -= int64_t(A);
    }
    const uint64_t r2 = uint64_t(r) * 2u;
    if (r2 > A || (r2 == A && (q & 1))) ++q;
    return q;
}

__device__ __forceinline__ int round_127_ratio(trit_u128 a, const IntMlpRow &R) {
    if (R.small) return round_127_ratio_small(uint64_t(a), uint64_t(R.A), R.k);
    const trit_u128 n = a * 127u;
    int q = 0;
#pragma unroll
    for (int b = 64; b; b >>= 1)
        if (trit_u128(q + b) * R.A <= n) q += b;
    const trit_u128 r = n - trit_u128(q) * R.A;
    if (2 * r > R.A || (2 * r == R.A && (q & 1))) ++q;
    return q;
}

// The signed code of one column.
__device__ __forceinline__ int intmlp_code(int32_t ag, int32_t au, const IntMlpRow &R) {
    if (R.zero) return 0;
    bool neg;
    const trit_u128 t = intmlp_abs_t(ag, au, neg);
    const int v = round_127_ratio(t, R);
    return neg ? -v : v;
}

// The same for a row with A < 2^56 (R.small, not R.zero): every |t| <= A fits
// 64 bits, so |t| is formed in 64-bit arithmetic.
__device__ __forceinline__ int intmlp_code_small(int32_t ag, int32_t au, const IntMlpRow &R) {
    if (ag <= 0 || au == 0) return 0;
    const uint64_t uu = au < 0 ? uint64_t(-int64_t(au)) : uint64_t(au);
    const uint64_t t = uint64_t(ag) * uint64_t(ag) * uu;
    const int v = round_127_ratio_small(t, uint64_t(R.A), R.k);
    return au < 0 ? -v : v;
}

// The signed code of one column, any row: an fp32 estimate first, the exact
// integer rounding only near a tie.  The estimate p = fl(fl(fl(g)^2) * fl(|u|)) * kf
// of 127 |t| / A carries at most ten fp32 roundings of relative size 2^-24
// (g twice through g^2, g^2, u, the product, A's two halves and their sum,
// 127 / fl(A), the last product), so |p - 127 |t| / A| <= 127 * 10 * 2^-24
// (1 + 2^-20) < 7.6e-5.  Where p's distance from the nearest half-integer
// exceeds 1.5e-4 the exact quotient lies on the same side of it and rounds to
// the same integer as p; otherwise the exact path decides.
//
// intmlp_code_fast has no branch: relu and the zero cases fall out of the
// arithmetic (g = 0 for a_g <= 0 gives p = 0; kf = 0 for a zero row), and p
// (0 <= p < 2^8) is rounded to an integer by adding and subtracting 1.5 * 2^23
// (fp32 round-to-nearest-even at unit spacing); fr = p - that integer is exact,
// and |fr| < 0.5 - 1.5e-4 is the "far from a tie" test.  Four columns then
// run as independent chains (intmlp_codes4) instead of four branchy calls.
// The exact path, kept out of line so that the unrolled column loops around
// it stay small.  R travels as scalars (by value, in registers).
static __device__ __noinline__ int intmlp_code_exact(int32_t ag, int32_t au, uint64_t a_hi,
                                                     uint64_t a_lo, float k, bool small) {
    IntMlpRow R;
    R.A = (trit_u128(a_hi) << 64) | trit_u128(a_lo);
    R.small = small;
    R.zero = false;
    R.k = k;
    R.kf = 0.0f;
    return small ? intmlp_code_small(ag, au, R) : intmlp_code(ag, au, R);
}

__device__ __forceinline__ int intmlp_code_fast(int32_t ag, int32_t au, const IntMlpRow &R,
                                                bool &near) {
    const float g = __int2float_rn(ag > 0 ? ag : 0);
    const float tf = __fmul_rn(__fmul_rn(g, g), fabsf(__int2float_rn(au)));
    const float p = __fmul_rn(tf, R.kf);
    const float big = __fadd_rn(p, 12582912.0f);
    const float fr = __fsub_rn(p, __fsub_rn(big, 12582912.0f));
    near = fabsf(fr) >= 0.49985f;
    int q = __float_as_int(big) - 0x4B400000;
    q = q > 127 ? 127 : q;
    return au < 0 ? -q : q;
}

__device__ __forceinline__ int intmlp_code_est(int32_t ag, int32_t au, const IntMlpRow &R) {
    bool near;
    const int q = intmlp_code_fast(ag, au, R, near);
    if (!near) return q;
    return intmlp_code_exact(ag, au, uint64_t(R.A >> 64), uint64_t(R.A), R.k, R.small);
}

// The same estimate from the column's signed fp32 product tf = fl(fl(g)^2) *
// fl(|u|) with u's sign (g = relu(a_g); 0 where the code is 0), formed by the
// producer with exactly intmlp_code_fast's operations, so p is the same.
__device__ __forceinline__ float intmlp_tf(int32_t ag, int32_t au) {
    const float g = __int2float_rn(ag > 0 ? ag : 0);
    const float tf = __fmul_rn(__fmul_rn(g, g), fabsf(__int2float_rn(au)));
    return au < 0 ? -tf : tf;
}
__device__ __forceinline__ int intmlp_code_tf(float tfs, const IntMlpRow &R, bool &near) {
    const float p = __fmul_rn(fabsf(tfs), R.kf);
    const float big = __fadd_rn(p, 12582912.0f);
    const float fr = __fsub_rn(p, __fsub_rn(big, 12582912.0f));
    near = fabsf(fr) >= 0.49985f;
    int q = __float_as_int(big) - 0x4B400000;
    q = q > 127 ? 127 : q;
    return tfs < 0.0f ? -q : q;
}

// Four columns' codes packed as bytes (column c in byte c).
__device__ __forceinline__ uint32_t intmlp_codes4(int4 g, int4 u, const IntMlpRow &R) {
    bool n0, n1, n2, n3;
    int c0 = intmlp_code_fast(g.x, u.x, R, n0);
    int c1 = intmlp_code_fast(g.y, u.y, R, n1);
    int c2 = intmlp_code_fast(g.z, u.z, R, n2);
    int c3 = intmlp_code_fast(g.w, u.w, R, n3);
    if (n0 | n1 | n2 | n3) {   // rare: a column within 1.5e-4 of a tie
        const uint64_t hi = uint64_t(R.A >> 64), lo = uint64_t(R.A);
        if (n0) c0 = intmlp_code_exact(g.x, u.x, hi, lo, R.k, R.small);
        if (n1) c1 = intmlp_code_exact(g.y, u.y, hi, lo, R.k, R.small);
        if (n2) c2 = intmlp_code_exact(g.z, u.z, hi, lo, R.k, R.small);
        if (n3) c3 = intmlp_code_exact(g.w, u.w, hi, lo, R.k, R.small);
    }
    return (uint32_t(c0) & 0xffu) | ((uint32_t(c1) & 0xffu) << 8) | ((uint32_t(c2) & 0xffu) << 16) |
           (uint32_t(c3) << 24);
}

// max|t| (hi:lo) * ((S_g * S_g) * S_u), S = w * x_scale / 127, in double, rounded once.
// Split in two so that the factor, which does not depend on max|t|, can be
// formed while max|t| is still being reduced.
__device__ __forceinline__ double intmlp_scale_factor(float w_g, float w_u, float x_scale) {
    const double s = double(x_scale);
    const double sg = __ddiv_rn(__dmul_rn(double(w_g), s), 127.0);
    const double su = __ddiv_rn(__dmul_rn(double(w_u), s), 127.0);
    return __dmul_rn(__dmul_rn(sg, sg), su);
}
__device__ __forceinline__ float intmlp_scale_apply(uint64_t hi, uint64_t lo, double k) {
    const double a = __dadd_rn(__dmul_rn(__ull2double_rn(hi), 18446744073709551616.0),
                               __ull2double_rn(lo));
    return __double2float_rn(__dmul_rn(a, k));
}
__device__ __forceinline__ float intmlp_scale(uint64_t hi, uint64_t lo, float w_g, float w_u,
                                              float x_scale) {
    return intmlp_scale_apply(hi, lo, intmlp_scale_factor(w_g, w_u, x_scale));
}

// The fp32 dequantisation of one output, one rounding per step, never contracted.
__device__ __forceinline__ float dequant(int32_t y, float w_scale, float x_scale) {
    float f = __int2float_rn(y);
    f = __fmul_rn(f, w_scale);
    f = __fmul_rn(f, x_scale);
    return div127_rn(f);
}

// Permuted activation layout used by the select-accumulate kernels.  For each
// 32-column half of a beat (h = 0: columns 0..31, h = 1: 32..63) word j (0..7)
// holds the bytes of columns 8i + j, i = 0..3, so that the four bits j, 8+j,
// 16+j, 24+j of a 32-bit plane word line up with its four bytes.  A beat takes
// 16 words; the shared-memory copy pads each beat to kXBeatWords words so that
// eight consecutive beats fall on distinct banks.
constexpr int kXBeatWords = 20;

// Transpose of one 32-column block: in[k] = natural words (bytes 4k..4k+3),
// out[j] = bytes (j, 8+j, 16+j, 24+j).
__device__ __forceinline__ void permute_block(const uint32_t in[8], uint32_t out[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int w = j >> 2;                  // word holding byte j within each 8-byte group
        const uint32_t s = (uint32_t)(j & 3);  // byte within that word
        // bytes: column j (word w), 8+j (word 2+w), 16+j (word 4+w), 24+j (word 6+w)
        uint32_t lo = prmt(in[w], in[2 + w], s | ((s + 4) << 4));
        uint32_t hi = prmt(in[4 + w], in[6 + w], s | ((s + 4) << 4));
        out[j] = prmt(lo, hi, 0x5410);
    }
}

// ---- activation quantiser arithmetic ------------------------------------------
// Shared by trit_quant_act and the fused quantise-and-multiply path so that both
// produce identical codes ("Tritium ..." -- Numerics; reading: q = clamp(rint(x *
// (127/a)), -127, 127) with a = max|x|, prescaled by 2^96 when a < 2^-96).

// |x| as an integer: non-negative floats order like their bit patterns.
__device__ __forceinline__ uint32_t quant_abs_bits(float v) { return __float_as_uint(v) & 0x7fffffffu; }

struct QuantScale {
    float a;      // the row's absmax (the stored x_scale), 0 for a zero or rejected row
    float pre;    // 2^96 when a < 2^-96, else 1
    float inv;    // 127 / (a * pre)
    bool zero;    // every code is 0
};

__device__ __forceinline__ QuantScale quant_scale(uint32_t amax_bits, bool bad) {
    QuantScale q;
    const float a = __uint_as_float(amax_bits);
    q.zero = bad || amax_bits == 0;
    q.a = q.zero ? 0.0f : a;
    q.pre = a < 0x1p-96f ? 0x1p96f : 1.0f;
    q.inv = q.zero ? 0.0f : __fdiv_rn(127.0f, __fmul_rn(a, q.pre));
    return q;
}

__device__ __forceinline__ int quant_code(float v, const QuantScale &q) {
    if (q.zero) return 0;
    int c = __float2int_rn(__fmul_rn(__fmul_rn(v, q.pre), q.inv));
    return c > 127 ? 127 : (c < -127 ? -127 : c);
}

__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d) {
    return (uint32_t(a) & 0xffu) | ((uint32_t(b) & 0xffu) << 8) | ((uint32_t(c) & 0xffu) << 16) |
           (uint32_t(d) << 24);
}

// ---- launchers (host) ---------------------------------------------------------

struct ProjDev {            // one product as a kernel sees it
    const uint4 *planes;
    const int8_t *x;        // int8 activations (unfused)
    const float *xf;        // fp32 activations (fused quantise-and-multiply), else NULL
    const float *x_scale;   // input scales (unfused) / output scale, may be NULL (fused)
    int8_t *x_i8_out;       // fused: output codes, may be NULL
    int32_t *y_i32;
    float *y_f32;
    int64_t M, N;
    int32_t K, B;
    float w_scale;
    float x_scale_val;      // the input scale when x_scale is NULL (M = 1 integer path only)
    bool planes_ready;      // TRIT_PROJ_PLANES_READY: planes may be read before the grid dependency
};

// One IntMlp down projection (M = 1): its activation row is formed in the
// launch from the gate and up projections' int32 outputs.  `down` carries the
// planes, the outputs (x_i8_out = the codes, x_scale = their scale, both
// optional), N, K, B and w_scale; its x and xf are NULL.
struct MlpProjDev {
    ProjDev down;
    const int32_t *a_gate, *a_up;
    const float *x_scale_in;
    float w_gate, w_up;
};
cudaError_t launch_intmlp_gemv_many(const MlpProjDev *list, int count, uint32_t *err,
                                    cudaStream_t s);

// One batch-1 MLP block for the two-launch path: gate and up (fp32 input,
// fused quantiser; y_i32 = a_gate / a_up, gate's x_scale = the input scale),
// the down projection (x_i8_out / x_scale = the optional h_i8 / h_scale
// outputs) and the per-CTA max|t| partials the gate/up launch publishes.
struct MlpBlockDev {
    ProjDev gate, up, down;
    float w_gate, w_up;
    uint64_t *tmax;   // 2 words (hi, lo) per partial
};
int64_t mlp_tmax_parts(int64_t F);
// The workspace of a block: mlp_tmax_parts(F) partials (hi, lo words), then
// 32 fp32 per partial: the signed products intmlp_tf of the partial's columns
// (0 past F).
inline int64_t mlp_tmax_bytes(int64_t F) { return mlp_tmax_parts(F) * (16 + 32 * 4); }
__host__ __device__ inline float *mlp_tf_of(uint64_t *tmax, int64_t parts) {
    return reinterpret_cast<float *>(tmax + 2 * parts);
}
bool mlp_pairs_supported(int64_t K, int64_t F);
cudaError_t launch_mlp_gate_up(const MlpBlockDev *list, int count, uint32_t *err, cudaStream_t s);
cudaError_t launch_mlp_down(const MlpBlockDev *list, int count, uint32_t *err, cudaStream_t s);

cudaError_t launch_pack(const int8_t *w, int64_t N, int64_t K, float w_scale, uint8_t *planes,
                        float *scale_out, uint32_t *err, cudaStream_t s);
cudaError_t launch_unpack(const uint8_t *planes, int64_t N, int64_t K, int8_t *w, uint32_t *err,
                          cudaStream_t s);
cudaError_t launch_verify(const uint8_t *planes, int64_t N, int64_t K, uint32_t *err,
                          unsigned long long *first_bad, cudaStream_t s);
cudaError_t launch_quant_many(const trit_act *list, int count, uint32_t *err, cudaStream_t s);

// M = 1 products (int8 activations, or fp32 activations quantised in the launch).
cudaError_t launch_gemv_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s);
// 2 <= M products, dp4a with beats reused across rows held in registers.
cudaError_t launch_gemm_dp4a_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s);

// kSkinnyMinM <= M <= kSkinnyMaxM (and K < 2^17, where fp32 accumulation of
// integer partial sums stays exact) runs on the tensor cores with the weights
// as the 128-row operand; larger M on CTA pairs with 256 x 256 tiles.
// measured on the 30-layer stack: the tensor cores take ~0.6 ms per step for
// any M up to 64, the dp4a path ~0.59 ms at M = 12 and 0.76 ms at M = 13..16
constexpr int64_t kSkinnyMinM = 13;
constexpr int64_t kSkinnyMaxM = 128;
bool skinny_supported(const ProjDev &p);
cudaError_t launch_skinny_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s);
// Bytes of the fp16 activation copy the small-M tensor-core path needs for p
// (128 * ceil(M/16)*16 * ceil(K/64): at most 32 MiB).
int64_t skinny_scratch_bytes(const ProjDev &p);
cudaError_t launch_skinny_into(const ProjDev &p, uint8_t *xh, uint32_t *err, cudaStream_t s);
constexpr int64_t kPrefillMinM = kSkinnyMaxM + 1;
bool prefill_supported(const ProjDev &p);
cudaError_t launch_prefill_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s);
// Bytes of the fp16 activation copy the tensor-core path needs for p.
int64_t prefill_scratch_bytes(const ProjDev &p);
// The tensor-core path for one product with its activation copy at xh
// (prefill_scratch_bytes(p) bytes, 16-byte aligned, caller-provided).
cudaError_t launch_prefill_into(const ProjDev &p, uint8_t *xh, uint32_t *err, cudaStream_t s);
// This device's fixed scratch buffer (TRIT_NOALLOC_SCRATCH_BYTES long).
cudaError_t fixed_scratch(uint8_t **out);
cudaError_t launch_quant_folded(const float *x, const float *g, int64_t M, int64_t K, float eps,
                                int8_t *q, float *x_scale, uint32_t *err, cudaStream_t s);
cudaError_t launch_read_probe(const void *p, int64_t bytes, uint32_t *sink, cudaStream_t s);
cudaError_t launch_issue_probe(int kind, int blocks, int threads, int64_t iters, uint32_t *sink,
                               unsigned long long *rec, cudaStream_t s);
cudaError_t launch_check_div127(uint64_t lo, uint64_t hi, unsigned long long *mismatches,
                                cudaStream_t s);
// max|t| partials of IntMlp blocks from their gate and up outputs: partial k of
// a block is max |relu(a_gate[c])^2 a_up[c]| over c in [32k, 32k + 32), the
// format the paired gate/up launch publishes (hi, lo words).
struct MlpTmaxJob {
    const int32_t *a_gate, *a_up;
    int64_t F;
    uint64_t *tmax;
};
cudaError_t launch_mlp_tmax(const MlpTmaxJob *jobs, int n, cudaStream_t s);
cudaError_t launch_intmlp_quant(const int32_t *ag, const int32_t *au, int64_t M, int64_t N,
                                float w_g, float w_u, const float *x_scale, int8_t *q,
                                float *h_scale, cudaStream_t s);

// BITCOS weights (presence bitmap + compacted signs), one activation row.
constexpr int64_t kBitcosMaxK = TRIT_BITCOS_MAX_K;
struct BitcosDev {
    const uint64_t *bitmap;
    const uint32_t *sign_off;
    const uint32_t *signs;
    const int8_t *x;
    const float *x_scale;
    int32_t *y_i32;
    float *y_f32;
    int64_t N, K, sign_words;
    float w_scale;
};
cudaError_t launch_bitcos_many(const BitcosDev *list, int count, cudaStream_t s);
// Host packer (trit_bitcos_pack): returns a trit_status.
int bitcos_pack_host(const int8_t *w, int64_t N, int64_t K, uint64_t *bitmap, uint32_t *sign_off,
                     uint32_t *signs, int64_t *sign_words);

int device_sm_count();

}  // namespace trit

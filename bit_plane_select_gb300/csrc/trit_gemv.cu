// Select-accumulate kernels for decode: y = W x over .trit v1 bit planes,
// exact int32 accumulation with dp4a, one persistent launch per product list.
//
// What is computed ("Tritium: One Weight Format for Ternary Inference ..." --
// Introduction, Eq. 3; "The .trit format, version 1" -- 1 and 2.3):
//   y_r = sum_{c : pos bit set} x_c - sum_{c : neg bit set} x_c
// over beats of 64 columns (pos, neg = two 64-bit masks).  Any beat with
// pos & neg != 0 sets TRIT_ERR_P1.
//
// Work split.  A warp handles 8 rows x 4 beats per step: lane = 4*rs + bs reads
// beat (4t + bs) of row (8g + rs) with one 16-byte load, so one warp load covers
// 8 x 64 contiguous bytes (whole 32-byte sectors).  A "group" is 8 rows; it
// takes ceil(B/4) steps.  The launch is persistent: every CTA gets an equal
// share of the total steps of the list (groups never split) and each warp a
// contiguous run of the CTA's groups; every entry's cost is preceded by a fixed
// staging charge, so CTAs that stage more entries get fewer groups.  The CTA
// keeps the activation row(s) of
// the current product in shared memory in the permuted layout of
// trit_internal.cuh.  Loads past the end of a warp's rows or of a row's beats
// are clamped to the last valid address (their data meets zero activations or
// an unwritten row), so the hot loop carries no predicates.
//
// M = 1 (two-bit codes, 4^j-weighted masks).  Column k of a beat gets the code
// c_k = 1 + pos_k - neg_k in {0, 1, 2}, so y = sum_k c_k x_k - sum_k x_k: the
// second sum is the activation row's own column sum, formed once while the
// row is staged.  Bit 1 of c_k is pos_k and bit 0 is NOR(pos_k, neg_k).  From
// the plane words P, N (32 columns) two words are built: ze holds the pairs
// (NOR_k, pos_k) of the even columns k at bits (k, k+1), zo those of the odd
// columns at bits (k-1, k) -- five logic instructions.  ze & (0x03030303 << 2j)
// then has byte i equal to 4^j c_k for column k = 8i + 2j (zo: 8i + 2j + 1),
// so one dp4a against the staged activation word of those columns covers both
// planes.  Eight accumulators, one per (j, parity), are divided by 4^j (exact:
// each is a multiple of 4^j) only when a row ends.  Cost per beat: 10 logic
// instructions to build the code words, then 16 AND + 16 dp4a.
//
// Long rows.  The staged activations must fit in shared memory, so a product
// whose rows exceed seg_beats(MT) beats is split into column segments.  Each
// segment adds its exact int32 partial into the output with an integer atomic
// (exact and order-independent, so the result is bit-identical to a single
// pass); the caller's int32 output, or else the fp32 output buffer read as
// int32, is zeroed first and a final pass applies the fp32 dequantisation.
// No scratch memory is used.
//
// Fused quantisation (M = 1).  An entry may carry its fp32 activation row
// instead of int8 codes: the CTA then quantises the row itself while staging
// it (the same arithmetic as trit_quant_act), so a whole decode token is one
// launch; the CTA that owns the entry's first group also writes the codes and
// the scale to global memory when asked.  The first plane loads of each warp
// are announced to L2 with a bulk prefetch before the staging barrier, so HBM
// streaming starts at once.
//
// Back-to-back launches.  Launches go out with programmatic stream
// serialisation: a launch that follows another one of these kernels may start
// while the first still runs (its CTAs take the SMs the first one frees), do
// its search and L2 prefetch, and wait for the first grid to finish before it
// reads activations or writes outputs -- the prefetch of the next token's
// planes overlaps the tail of the current one.
//
// M > 1 (masked code words).  Each beat's code words are formed once (the M = 1
// code words) and masked into sixteen words of bytes 4^k c, c in {0, 1, 2},
// reused for every activation row held by the CTA: 16 dp4a per row into one of
// NJ accumulators per weight class k (NJ = 4: 16 AND per beat, no shift; NJ = 1:
// code bytes of weight 1, 28 logic instructions per beat), folded exactly at
// the row's end, then the row's column sum is subtracted.  A lane
// holds two weight rows (16-row groups), so every activation word it reads
// from shared memory serves two rows; the CTA stages its MT activation rows
// beat-interleaved (all rows of a beat side by side) so every read is an
// immediate offset from one pointer.  At a group's end the four lanes of a row
// set reduce-scatter their partial sums, so every row is finished by two of
// them and stored by one.  The
// bound is the dp4a rate: 64 lanes per SM-clock on this device, i.e. two
// SM-clocks per row-beat at M = 8 (the probe in trit_probe.cu measures it).
#include "trit_internal.cuh"

namespace trit {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// Lanes per weight row: M > 1 paths 4; M = 1 TRIT_M1_LANES (4: a warp load
// covers 8 rows x 64 bytes; 8: 4 rows x 128 bytes).  A plain read probe of the
// stack's rows streams 3-5% faster with 4 x 128 bytes, but the kernel is
// slower with it: 100.2 against 95.8 us per 30-layer token (ring depth 2, 7
// and 14 for the 108-beat rows, two or four groups prefetched: all slower).
#ifndef TRIT_M1_LANES
#define TRIT_M1_LANES 4
#endif
constexpr int kLanesPerRow = 4;
constexpr int kLanes1 = TRIT_M1_LANES;
static_assert(kLanes1 == 4 || kLanes1 == 8, "lanes per row at M = 1");
constexpr int kRowsPerGroup = 32 / kLanes1;   // rows of an M = 1 group
__host__ __device__ constexpr int lanes_of(int mt) { return mt == 1 ? kLanes1 : kLanesPerRow; }
// The unrolled M = 1 paths: rows of 40 and 108 beats (K = 2560, 6912).
constexpr int kIt40 = 40 / kLanes1;
constexpr int kIt108 = (108 + kLanes1 - 1) / kLanes1;
constexpr int kDepth = 4;                   // 16-byte loads in flight per lane
constexpr int kMaxList = TRIT_MAX_LIST_PER_LAUNCH;
constexpr int kXBeatVec = kXBeatWords / 4;  // uint4 per staged beat

// Groups ahead of the one being computed that each warp bulk-prefetches into
// L2 (0 disables: measured slower at every distance on the 30-layer stack),
// how many of the first groups of each warp are prefetched before the staging
// barrier, and the register ring depths of the unrolled paths (measured: depth
// matters little once 24 warps per SM are resident).
#ifndef TRIT_L2_AHEAD
#define TRIT_L2_AHEAD 0
#endif
#ifndef TRIT_RING_40
#define TRIT_RING_40 5
#endif
#ifndef TRIT_RING_108
#define TRIT_RING_108 (TRIT_M1_LANES == 8 ? 7 : 3)
#endif
#ifndef TRIT_PREFETCH_FIRST
#define TRIT_PREFETCH_FIRST (TRIT_M1_LANES == 8 ? 4 : 2)
#endif
#ifndef TRIT_COST_108
#define TRIT_COST_108 100
#endif
#ifndef TRIT_WAVES
#define TRIT_WAVES 1
#endif
#ifndef TRIT_MIN_BLOCKS_M1
#define TRIT_MIN_BLOCKS_M1 3
#endif
// M > 1 path: steps of loads in flight per row of a lane, per staged row count.
#ifndef TRIT_RING_M2
#define TRIT_RING_M2 4
#endif
#ifndef TRIT_RING_M4
#define TRIT_RING_M4 4
#endif
#ifndef TRIT_RING_M8
#define TRIT_RING_M8 2
#endif
__host__ __device__ constexpr int ring_rows(int mt) {
    return mt == 8 ? TRIT_RING_M8 : mt == 4 ? TRIT_RING_M4 : TRIT_RING_M2;
}
// M > 1 path: accumulators per (weight row, activation row) -- the number of
// weight classes 4^j the code words are masked into (4: every mask is an AND of
// the code word, no shift; 2: one shift per code word; 1: code bytes of weight
// 1, three shifts per code word) -- per staged row count.  Measured on the
// 30-layer stack with four weight rows per lane: M = 2 129.9 us with 1 class,
// 123.6 with 2, 121.5 with 4; M = 4 unchanged by 2 classes (4 spill); M = 8
// spilled with 2 (351 against 322 us).  With two rows per lane (below) M = 8
// takes 2 classes without spilling.
#ifndef TRIT_NJ_M2
#define TRIT_NJ_M2 4
#endif
#ifndef TRIT_NJ_M4
#define TRIT_NJ_M4 2
#endif
#ifndef TRIT_NJ_M8
#define TRIT_NJ_M8 2
#endif
__host__ __device__ constexpr int acc_classes(int mt) {
    return mt == 8 ? TRIT_NJ_M8 : mt == 4 ? TRIT_NJ_M4 : TRIT_NJ_M2;
}
// CTAs per SM the kernel is compiled for (its register budget: 128 per thread
// for MT > 1)
#ifndef TRIT_MIN_BLOCKS_M2
#define TRIT_MIN_BLOCKS_M2 2
#endif
__host__ __device__ constexpr int min_blocks(int mt) {
    return mt == 1 ? TRIT_MIN_BLOCKS_M1 : mt == 2 ? TRIT_MIN_BLOCKS_M2 : 2;
}
// Cost units charged ahead of each entry's groups for staging its activations
// (M = 1 launches; a group step costs 100; 0 disables): a CTA whose share starts
// an entry gets that much less group work.  Measured on the 30-layer stack (3,000 ... 70,000
// swept): 30,000 (the time of ~11 average CTA group-steps per warp) is best.
#ifndef TRIT_STAGE_COST
#define TRIT_STAGE_COST 30000
#endif
constexpr int64_t kStageCost = TRIT_STAGE_COST;
// The same charge for launches staging MT > 1 rows (a group step there is a
// 32-row group's step; 0 disables).  Measured on the 30-layer stack: 8,000
// takes M = 8 from 322.9 to 312.7 us and M = 4 from 191.0 to 188.1 us, and costs
// M = 2 three microseconds, so two-row launches take none.
#ifndef TRIT_STAGE_COST_M2
#define TRIT_STAGE_COST_M2 0
#endif
#ifndef TRIT_STAGE_COST_MT
#define TRIT_STAGE_COST_MT 8000
#endif
__host__ __device__ constexpr int64_t stage_cost(int mt) {
    return mt == 1 ? kStageCost : mt == 2 ? int64_t(TRIT_STAGE_COST_M2) : int64_t(TRIT_STAGE_COST_MT);
}
constexpr int kL2Ahead = TRIT_L2_AHEAD;

// Beats per column segment for MT staged rows: MT * seg_beats * 80 bytes of
// shared memory stay at 90 KB.  A segment takes at most 288 steps per row, so
// the 4^j-weighted accumulators (at most 2^17 per step) stay below 2^26.
__host__ __device__ constexpr int seg_beats(int mt) { return 1152 / mt; }

struct Entry {
    const uint4 *planes;
    const int8_t *x;        // first activation row of this entry, stride xld
    const float *xf;        // fused: the fp32 activation row (x is unused)
    int8_t *x_i8_out;       // fused: codes out (natural layout, K_pad bytes), may be NULL
    const float *x_scale;   // first scale of this entry (fused: scale out, may be NULL)
    int32_t *y_i32;         // first output row of this entry, stride N
    float *y_f32;
    int32_t *acc;           // non-NULL: atomically add the int32 partial here (stride N)
    int64_t N;
    int64_t groups;         // ceil(N / 8)
    int64_t cost_begin;     // prefix sum of groups * gcost over the list
    int32_t xld;            // activation row stride (K_pad)
    int32_t K, B, iters;    // columns and beats of this entry's segment; iters = ceil(B / lanes)
    int32_t bstride;        // beats per full row of the planes
    int32_t mrows;          // bits 0-7: activation rows of this entry (<= MT); bits 8-15:
                            // 1 + index of its IntMlp descriptor (0: none); bit 16:
                            // kPlanesReady
    int32_t gcost;          // cost units of one group: iters x a per-step weight
    float w_scale;
};
static_assert(sizeof(Entry) == 120, "the list of 256 entries must fit the 32 KB parameter space");

// An IntMlp input (M = 1): the entry's activation row is formed from the int32
// outputs of the gate and up projections of the same token.
struct MlpDesc {
    const int32_t *a_gate, *a_up;   // [K] each
    const float *x_scale;           // the gate/up input's activation scale
    float w_gate, w_up;
    // pre-loading launches: the per-CTA max|t| partials (hi, lo word pairs) a
    // paired gate/up launch writes and the down launch reduces
    uint64_t *tmax;
    int32_t ntmax;
    int32_t pad_;
};
constexpr int kMaxMlp = 8;   // IntMlp descriptors per launch (each adds 48 bytes to every launch's parameters)

struct List {
    int32_t count;
    int32_t xs_words;       // shared words of the staged activations
    int64_t total_cost;
    uint32_t *err;
    float x_scale_val;      // M = 1 entries whose x_scale is NULL take this input scale
    int32_t flags;          // pre-loading launches: 1 = copy the planes before the grid
                            // dependency, 2 = paired gate/up list, 4 = two warps per group
    int32_t plane_steps;    // pre-loading launches: 16-byte plane slots per lane
    int32_t pad_;
    MlpDesc mlp[kMaxMlp];
    Entry e[kMaxList];
};
static_assert(sizeof(List) <= 32764, "kernel parameter space");

__host__ __device__ __forceinline__ int rows_of(const Entry &E) { return E.mrows & 0xff; }
__host__ __device__ __forceinline__ int mlp_of(const Entry &E) { return (E.mrows >> 8) & 0xff; }
// Entry.mrows bit: the planes may be read before the grid dependency resolves
constexpr int32_t kPlanesReady = 1 << 16;

// Code-word multiply-accumulate of one 32-column plane word pair (M = 1).
__device__ __forceinline__ void mac_codes(uint32_t P, uint32_t N, const uint32_t (&x)[8],
                                          int (&acc)[8]) {
    const uint32_t nor = ~(P | N);
    const uint32_t ze = (nor & 0x55555555u) | ((P << 1) & 0xAAAAAAAAu);
    const uint32_t zo = ((nor >> 1) & 0x55555555u) | (P & 0xAAAAAAAAu);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t m = 0x03030303u << (2 * j);
        acc[j] = dp4a_su(x[2 * j], ze & m, acc[j]);
        acc[4 + j] = dp4a_su(x[2 * j + 1], zo & m, acc[4 + j]);
    }
}

// sum_k c_k x_k of a lane from its eight 4^j-weighted accumulators.
__device__ __forceinline__ int32_t codes_total(const int (&acc)[8]) {
    return (acc[0] + acc[4]) + ((acc[1] + acc[5]) >> 2) + ((acc[2] + acc[6]) >> 4) +
           ((acc[3] + acc[7]) >> 6);
}

// Column sum of the staged activation row (M = 1): each warp publishes its
// part; every thread adds the parts after the staging barrier.
__device__ __forceinline__ void publish_xsum(int32_t v, int32_t *s_xsum) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
    if ((threadIdx.x & 31) == 0) s_xsum[threadIdx.x >> 5] = v;
}
__device__ __forceinline__ int32_t read_xsum(const int32_t *s_xsum) {
    int32_t s = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) s += s_xsum[i];
    return s;
}
// Column sum of staged row m of MT (the parts of the warps that staged it).
template <int MT>
__device__ __forceinline__ int32_t read_xsum_row(const int32_t *s_xsum, int m) {
    constexpr int kWpr = kWarps / MT;
    int32_t s = 0;
#pragma unroll
    for (int i = 0; i < kWpr; ++i) s += s_xsum[m * kWpr + i];
    return s;
}

// Two-bit code words of one 32-column plane word pair (P, N): ze holds the
// codes c = 1 + pos - neg in {0, 1, 2} of the even columns k at bits (k, k+1),
// zo those of the odd columns at bits (k-1, k), so (ze >> 2j) & 0x03030303 has
// byte i = c of column 8i + 2j and (zo >> 2j) & 0x03030303 that of column
// 8i + 2j + 1 -- the columns of staged activation words 2j and 2j + 1.
__device__ __forceinline__ void code_words(uint32_t P, uint32_t N, uint32_t &ze, uint32_t &zo) {
    const uint32_t nor = ~(P | N);
    ze = (nor & 0x55555555u) | ((P << 1) & 0xAAAAAAAAu);
    zo = ((nor >> 1) & 0x55555555u) | (P & 0xAAAAAAAAu);
}

// Shared-memory words of one staged beat.  M = 1: the row's beats at a stride
// of kXBeatWords.  MT > 1: the MT rows' words of a beat side by side (16 words
// each: the two permuted 32-column halves), beats at a stride of MT * 16 + 4
// words -- 4 words mod 32 banks, so the four beats a warp reads at once fall on
// distinct banks -- and every row's words of a beat at a fixed offset from the
// beat's start, so the product loop addresses them with immediate offsets.
__host__ __device__ constexpr int beat_words(int mt) { return mt == 1 ? kXBeatWords : mt * 16 + 4; }
template <int MT>
__device__ __forceinline__ int xs_word(int m, int beat) {
    return MT == 1 ? beat * kXBeatWords : beat * beat_words(MT) + m * 16;
}

// Stage activation rows 0..MT-1 of entry E into shared memory, permuted, zero
// past column K and for rows >= mrows, covering iters*4 beats.  Row m is
// staged by warps m*kWarps/MT .. (m+1)*kWarps/MT - 1, each of which publishes
// its part of the row's column sum in s_xsum[warp].
template <int MT>
__device__ __forceinline__ void stage_x(const Entry &E, uint32_t *xs, int32_t *s_xsum) {
    static_assert(kWarps % MT == 0, "whole warps per staged row");
    constexpr int kWpr = kWarps / MT;
    const int halves = E.iters * lanes_of(MT) * 2;
    const int m = (threadIdx.x >> 5) / kWpr;
    int32_t xsum = 0;
    for (int hb = ((threadIdx.x >> 5) % kWpr) * 32 + (threadIdx.x & 31); hb < halves;
         hb += kWpr * 32) {
        uint32_t out[8];
        if (m < rows_of(E)) {
            const int c0 = hb * 32;
            const int8_t *xr = E.x + int64_t(m) * E.xld;
            uint32_t in[8];
            if (c0 + 32 <= E.K) {
                const uint4 *p = reinterpret_cast<const uint4 *>(xr + c0);
                const uint4 u0 = p[0], u1 = p[1];
                in[0] = u0.x; in[1] = u0.y; in[2] = u0.z; in[3] = u0.w;
                in[4] = u1.x; in[5] = u1.y; in[6] = u1.z; in[7] = u1.w;
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t w = 0;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int c = c0 + 4 * k + b;
                        const uint32_t v = c < E.K ? (uint32_t)(uint8_t)xr[c] : 0u;
                        w |= v << (8 * b);
                    }
                    in[k] = w;
                }
            }
            permute_block(in, out);
#pragma unroll
            for (int k = 0; k < 8; ++k) xsum = dp4a_ss(in[k], 0x01010101u, xsum);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) out[j] = 0;
        }
        uint32_t *dst = xs + xs_word<MT>(m, hb >> 1) + (hb & 1) * 8;
        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
    publish_xsum(xsum, s_xsum);
}

// Fused path: quantise the fp32 row of entry E (K <= seg_beats(1)*64 columns)
// straight into the permuted shared-memory layout, with the arithmetic of
// trit_quant_act.  Each thread owns 4-column quads q = tid, tid + 256, ...;
// the first kHoldQ of them stay in registers between the absmax pass and the
// code pass (the rest are re-read, from L1).  A quad's four codes land in four
// permuted words of its 32-column half-block (column 8i + j -> word j, byte i).
// The owner CTA also writes the natural-layout codes (zero tail to K_pad) and
// the scale.  Returns the scale.
constexpr int kHoldQ = 4;
// The four codes w (bytes: columns 4q..4q+3) into the permuted layout: column
// 8i + j of a 32-column half-block goes to word j, byte i.  (Byte stores: a
// variant gathering whole words with four warp shuffles per lane measured
// slower.)
__device__ __forceinline__ void put_quad(uint32_t *xs, int q, uint32_t w) {
    const int hb = q >> 3, k = q & 7;
    uint8_t *dst = reinterpret_cast<uint8_t *>(xs + (hb >> 1) * kXBeatWords + (hb & 1) * 8 +
                                               4 * (k & 1)) + (k >> 1);
    dst[0] = uint8_t(w);
    dst[4] = uint8_t(w >> 8);
    dst[8] = uint8_t(w >> 16);
    dst[12] = uint8_t(w >> 24);
}
__device__ __forceinline__ float stage_x_fp32(const Entry &E, uint32_t *xs, bool owner,
                                              uint32_t *err, int32_t *s_xsum) {
    __shared__ uint32_t s_red[2][kWarps];
    const int K = E.K;
    const int nq = (K + 3) / 4;                  // quads that hold columns
    const int sq = E.iters * kLanes1 * 16;       // quads staged (>= nq)
    const float *x = E.xf;
    const bool vec = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(x) & 15) == 0);
    auto load4 = [&](int q) -> float4 {   // columns 4q..4q+3, zero past K
        const int c = 4 * q;
        if (vec && c + 4 <= K) return *reinterpret_cast<const float4 *>(x + c);
        float4 f;
        f.x = c + 0 < K ? x[c + 0] : 0.0f;
        f.y = c + 1 < K ? x[c + 1] : 0.0f;
        f.z = c + 2 < K ? x[c + 2] : 0.0f;
        f.w = c + 3 < K ? x[c + 3] : 0.0f;
        return f;
    };
    uint32_t amax = 0, bad = 0;
    auto scan = [&](const float4 &f) {
        bad |= !isfinite(f.x) | !isfinite(f.y) | !isfinite(f.z) | !isfinite(f.w);
        amax = max(amax, max(max(quant_abs_bits(f.x), quant_abs_bits(f.y)),
                             max(quant_abs_bits(f.z), quant_abs_bits(f.w))));
    };
    float4 held[kHoldQ];
#pragma unroll
    for (int r = 0; r < kHoldQ; ++r) {
        const int q = int(threadIdx.x) + r * kThreads;
        held[r] = q < nq ? load4(q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int r = 0; r < kHoldQ; ++r) scan(held[r]);
    for (int q = int(threadIdx.x) + kHoldQ * kThreads; q < nq; q += kThreads) scan(load4(q));
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        amax = max(amax, __shfl_xor_sync(~0u, amax, o));
        bad |= __shfl_xor_sync(~0u, bad, o);
    }
    if ((threadIdx.x & 31) == 0) {
        s_red[0][threadIdx.x >> 5] = amax;
        s_red[1][threadIdx.x >> 5] = bad;
    }
    __syncthreads();
    amax = 0;
    bad = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
        amax = max(amax, s_red[0][i]);
        bad |= s_red[1][i];
    }
    const QuantScale qs = quant_scale(amax, bad != 0);
    const int64_t Kp = beats_per_row(K) * 64;
    int32_t xsum = 0;
    auto emit = [&](int q, const float4 &f) {
        const uint32_t w = pack4(quant_code(f.x, qs), quant_code(f.y, qs), quant_code(f.z, qs),
                                 quant_code(f.w, qs));
        xsum = dp4a_ss(w, 0x01010101u, xsum);
        if (owner && E.x_i8_out && int64_t(q) * 4 < Kp)
            *reinterpret_cast<uint32_t *>(E.x_i8_out + int64_t(q) * 4) = w;
        put_quad(xs, q, w);
    };
#pragma unroll
    for (int r = 0; r < kHoldQ; ++r) {
        const int q = int(threadIdx.x) + r * kThreads;
        if (q < sq) emit(q, held[r]);
    }
    for (int q = int(threadIdx.x) + kHoldQ * kThreads; q < sq; q += kThreads)
        emit(q, q < nq ? load4(q) : make_float4(0.f, 0.f, 0.f, 0.f));
    publish_xsum(xsum, s_xsum);
    if (owner && threadIdx.x == 0) {
        if (E.x_scale) *const_cast<float *>(E.x_scale) = qs.a;
        if (bad) atomicOr(err, TRIT_ERR_NONFINITE);
    }
    return qs.a;
}

// IntMlp input (M = 1): the codes of t = relu(a_gate)^2 a_up for the row of
// entry E, round-half-even(127 t / max|t|), straight into the permuted
// shared-memory layout, with the arithmetic of trit_intmlp_quant.  Pass 1 finds
// max|t| (one block reduction), pass 2 forms the codes (the second read of a_gate
// and a_up hits L1).  The owner CTA also writes the natural-layout codes (zero
// tail to K_pad) and the scale.  The scale goes to *s_scale (shared), readable
// after the staging barrier.
__device__ __forceinline__ void stage_x_intmlp(const Entry &E, const MlpDesc &D, uint32_t *xs,
                                               bool owner, int32_t *s_xsum, float *s_scale) {
    __shared__ uint64_t s_max[2][kWarps];
    const int K = E.K;
    const int halves = E.iters * kLanes1 * 2;
    // 16-byte loads when the rows allow them (K % 4 == 0, 16-byte aligned)
    const bool vec = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(D.a_gate) & 15) == 0) &&
                     ((reinterpret_cast<uintptr_t>(D.a_up) & 15) == 0);
    trit_u128 amax = 0;
    auto take = [&](int32_t g, int32_t u) {
        bool neg;
        const trit_u128 t = intmlp_abs_t(g, u, neg);
        amax = t > amax ? t : amax;
    };
    // rounds of four loads per thread and array, issued together (the loads are
    // predicated, not behind loop exits)
    if (vec) {
        const int4 *G = reinterpret_cast<const int4 *>(D.a_gate);
        const int4 *U = reinterpret_cast<const int4 *>(D.a_up);
        const int K4 = K / 4;
        for (int base = 0; base < K4; base += 4 * kThreads) {
            int4 g[4], u[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = base + r * kThreads + threadIdx.x;
                g[r] = i < K4 ? G[i] : make_int4(0, 0, 0, 0);
                u[r] = i < K4 ? U[i] : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                take(g[r].x, u[r].x);
                take(g[r].y, u[r].y);
                take(g[r].z, u[r].z);
                take(g[r].w, u[r].w);
            }
        }
    } else {
        for (int base = 0; base < K; base += 4 * kThreads) {
            int32_t g[4], u[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int c = base + r * kThreads + threadIdx.x;
                g[r] = c < K ? D.a_gate[c] : 0;
                u[r] = c < K ? D.a_up[c] : 0;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) take(g[r], u[r]);
        }
    }
    uint64_t hi = uint64_t(amax >> 64), lo = uint64_t(amax);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const uint64_t h2 = __shfl_xor_sync(~0u, hi, o), l2 = __shfl_xor_sync(~0u, lo, o);
        if (h2 > hi || (h2 == hi && l2 > lo)) {
            hi = h2;
            lo = l2;
        }
    }
    if ((threadIdx.x & 31) == 0) {
        s_max[0][threadIdx.x >> 5] = hi;
        s_max[1][threadIdx.x >> 5] = lo;
    }
    __syncthreads();
    hi = s_max[0][0];
    lo = s_max[1][0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i)
        if (s_max[0][i] > hi || (s_max[0][i] == hi && s_max[1][i] > lo)) {
            hi = s_max[0][i];
            lo = s_max[1][i];
        }
    const IntMlpRow R = intmlp_row(hi, lo);
    const int64_t Kp = beats_per_row(K) * 64;
    int32_t xsum = 0;
    for (int hb = threadIdx.x; hb < halves; hb += kThreads) {
        const int c0 = hb * 32;
        const bool full = vec && c0 + 32 <= K;
        uint32_t in[8];
#pragma unroll
        for (int h8 = 0; h8 < 4; ++h8) {   // eight columns at a time
            int32_t g[8], u[8];
            const int cb = c0 + 8 * h8;
            if (full) {
                const int4 *G = reinterpret_cast<const int4 *>(D.a_gate + cb);
                const int4 *U = reinterpret_cast<const int4 *>(D.a_up + cb);
                const int4 a0 = G[0], a1 = G[1], b0 = U[0], b1 = U[1];
                g[0] = a0.x; g[1] = a0.y; g[2] = a0.z; g[3] = a0.w;
                g[4] = a1.x; g[5] = a1.y; g[6] = a1.z; g[7] = a1.w;
                u[0] = b0.x; u[1] = b0.y; u[2] = b0.z; u[3] = b0.w;
                u[4] = b1.x; u[5] = b1.y; u[6] = b1.z; u[7] = b1.w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const bool ok = cb + j < K;
                    g[j] = ok ? D.a_gate[cb + j] : 0;   // a zero gate output gives code 0
                    u[j] = ok ? D.a_up[cb + j] : 0;
                }
            }
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                int v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c = 4 * w + j;
                    v[j] = intmlp_code_est(g[c], u[c], R);
                }
                in[2 * h8 + w] = pack4(v[0], v[1], v[2], v[3]);
                xsum = dp4a_ss(in[2 * h8 + w], 0x01010101u, xsum);
            }
        }
        if (owner && E.x_i8_out && int64_t(hb) * 32 < Kp) {
            uint4 *o = reinterpret_cast<uint4 *>(E.x_i8_out + int64_t(hb) * 32);
            o[0] = make_uint4(in[0], in[1], in[2], in[3]);
            o[1] = make_uint4(in[4], in[5], in[6], in[7]);
        }
        uint32_t out[8];
        permute_block(in, out);
        uint32_t *dst = xs + (hb >> 1) * kXBeatWords + (hb & 1) * 8;
        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
    publish_xsum(xsum, s_xsum);
    // the scale (double arithmetic, slow on this device) by one thread; the
    // others read it after the staging barrier
    if (threadIdx.x == 0) {
        const float scale = intmlp_scale(hi, lo, D.w_gate, D.w_up, *D.x_scale);
        *s_scale = scale;
        if (owner && E.x_scale) *const_cast<float *>(E.x_scale) = scale;
    }
}

// 16-byte asynchronous copy global -> shared (cached in L2 only); completes at
// the issuing thread's cpa_wait_all, visible to that thread.
__device__ __forceinline__ void cpa16(void *smem, const void *gmem) {
    const uint32_t sa = uint32_t(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cpa_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// IntMlp input of a pre-loading launch (M = 1): as stage_x_intmlp, but max|t|
// is reduced from the D.ntmax per-CTA partials the gate/up launch published,
// and each column's code starts from the signed fp32 product it published
// beside them (intmlp_tf), so the row is read once and as 4 bytes a column:
// the products are copied into shared memory (rows: iters x 256 fp32) with
// every copy in flight together with the partials' loads, and the codes follow
// the reduction; a column near a tie reads its a_gate and a_up for the exact
// path.  The last thread forms the scale (its double-precision factor while
// the loads are in flight); the scale goes to *s_scale, readable after the
// staging barrier.  The owner CTA also writes the natural-layout codes (zero
// tail to K_pad) and the scale.
__device__ __forceinline__ void stage_x_intmlp_parts(const Entry &E, const MlpDesc &D, uint32_t *xs,
                                                     int32_t *rows, bool owner, int32_t *s_xsum,
                                                     float *s_scale) {
    __shared__ uint64_t s_m[2][kWarps];
    const int K = E.K;
    const int nq = (K + 3) / 4, sq = E.iters * kLanes1 * 16;
    float *st = reinterpret_cast<float *>(rows);
    // the products buffer holds 32 values per partial (zero past K): whole quads
    const float *tfg = mlp_tf_of(D.tmax, D.ntmax);
    for (int q = threadIdx.x; q < nq; q += kThreads) cpa16(st + 4 * q, tfg + 4 * q);
    cpa_commit();
    const bool scaler = threadIdx.x == kThreads - 1;
    uint64_t hi = 0, lo = 0;
    auto umax = [&](uint64_t h2, uint64_t l2) {
        if (h2 > hi || (h2 == hi && l2 > lo)) {
            hi = h2;
            lo = l2;
        }
    };
    for (int i = threadIdx.x; i < D.ntmax; i += kThreads) umax(D.tmax[2 * i], D.tmax[2 * i + 1]);
    // the scale's factor while the partials' loads are in flight
    double kfac = 0.0;
    if (scaler) kfac = intmlp_scale_factor(D.w_gate, D.w_up, *D.x_scale);
#pragma unroll
    for (int o = 16; o; o >>= 1) umax(__shfl_xor_sync(~0u, hi, o), __shfl_xor_sync(~0u, lo, o));
    if ((threadIdx.x & 31) == 0) {
        s_m[0][threadIdx.x >> 5] = hi;
        s_m[1][threadIdx.x >> 5] = lo;
    }
    cpa_wait_all();
    __syncthreads();   // the partials' maxima and every copied product
#pragma unroll
    for (int i = 0; i < kWarps; ++i) umax(s_m[0][i], s_m[1][i]);
    const IntMlpRow R = intmlp_row(hi, lo);
    const int64_t Kp = beats_per_row(K) * 64;
    int32_t xsum = 0;
    for (int q = threadIdx.x; q < sq; q += kThreads) {
        const float4 f = q < nq ? *reinterpret_cast<const float4 *>(st + 4 * q)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        bool n0, n1, n2, n3;
        int c0 = intmlp_code_tf(f.x, R, n0), c1 = intmlp_code_tf(f.y, R, n1);
        int c2 = intmlp_code_tf(f.z, R, n2), c3 = intmlp_code_tf(f.w, R, n3);
        if (n0 | n1 | n2 | n3) {   // rare: a column within 1.5e-4 of a tie (never past K)
            const int c = 4 * q;
            const uint64_t ah = uint64_t(R.A >> 64), al = uint64_t(R.A);
            if (n0) c0 = intmlp_code_exact(D.a_gate[c], D.a_up[c], ah, al, R.k, R.small);
            if (n1) c1 = intmlp_code_exact(D.a_gate[c + 1], D.a_up[c + 1], ah, al, R.k, R.small);
            if (n2) c2 = intmlp_code_exact(D.a_gate[c + 2], D.a_up[c + 2], ah, al, R.k, R.small);
            if (n3) c3 = intmlp_code_exact(D.a_gate[c + 3], D.a_up[c + 3], ah, al, R.k, R.small);
        }
        const uint32_t w = pack4(c0, c1, c2, c3);
        xsum = dp4a_ss(w, 0x01010101u, xsum);
        if (owner && E.x_i8_out && int64_t(q) * 4 < Kp)
            *reinterpret_cast<uint32_t *>(E.x_i8_out + int64_t(q) * 4) = w;
        put_quad(xs, q, w);
    }
    publish_xsum(xsum, s_xsum);
    if (scaler) {
        const float scale = intmlp_scale_apply(hi, lo, kfac);
        *s_scale = scale;
        if (owner && E.x_scale) *const_cast<float *>(E.x_scale) = scale;
    }
}

__device__ __forceinline__ int32_t row_sum1(int32_t v) {
    v += __shfl_xor_sync(~0u, v, 1);
    v += __shfl_xor_sync(~0u, v, 2);
    if (kLanes1 == 8) v += __shfl_xor_sync(~0u, v, 4);
    return v;
}

// M = 1, any row length: process groups [gb, ge) of entry E with one warp.
// Returns the OR of pos & neg.
__device__ __forceinline__ uint32_t run_groups(const Entry &E, const uint32_t *xs, float xsc,
                                               int32_t xsum, int64_t gb, int64_t ge, int rs,
                                               int bs) {
    const int it = E.iters;
    const int steps = int(ge - gb) * it;
    const int64_t N = E.N;
    uint32_t viol = 0;

    // ---- load cursor: beat loff of the (clamped) row at lrow; loff runs
    // bs, bs+4, ... and is clamped to the row's last beat, rows past the warp's
    // last valid row read that row -- every load stays inside the planes
    const int last_beat = E.B - 1;
    const int64_t last_row = (ge * kRowsPerGroup < N ? ge * kRowsPerGroup : N) - 1;
    int64_t lrow_idx = gb * kRowsPerGroup + rs;
    const uint4 *lrow = E.planes + (lrow_idx < last_row ? lrow_idx : last_row) * E.bstride;
    int lt = 0, loff = bs;
    auto next_load = [&]() -> uint4 {
        const uint4 v = ldg_stream(lrow + (loff < last_beat ? loff : last_beat));
        loff += kLanes1;
        if (++lt == it) {
            lt = 0;
            loff = bs;
            lrow_idx += kRowsPerGroup;
            lrow = E.planes + (lrow_idx < last_row ? lrow_idx : last_row) * E.bstride;
        }
        return v;
    };

    uint4 ring[kDepth];
#pragma unroll
    for (int d = 0; d < kDepth; ++d) ring[d] = next_load();

    // ---- compute cursor
    int acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0;
    int64_t row = gb * kRowsPerGroup + rs;
    int ct = 0;
    const uint4 *xs4 = reinterpret_cast<const uint4 *>(xs);
    const int xbase = bs * kXBeatVec;
    int xoff = xbase;

    auto body = [&](uint4 &slot) {
        const uint4 v = slot;
        slot = next_load();
        viol |= (v.x & v.z) | (v.y & v.w);
        const uint4 a0 = xs4[xoff], a1 = xs4[xoff + 1], a2 = xs4[xoff + 2], a3 = xs4[xoff + 3];
        const uint32_t xl[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const uint32_t xh[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
        mac_codes(v.x, v.z, xl, acc);
        mac_codes(v.y, v.w, xh, acc);
        xoff += kLanes1 * kXBeatVec;
        if (++ct == it) {
            const int32_t y = row_sum1(codes_total(acc)) - xsum;
            if (bs == 0 && row < N) {
                if (E.acc) {
                    atomicAdd(E.acc + row, y);
                } else {
                    if (E.y_i32) E.y_i32[row] = y;
                    if (E.y_f32) E.y_f32[row] = dequant(y, E.w_scale, xsc);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = 0;
            ct = 0;
            xoff = xbase;
            row += kRowsPerGroup;
        }
    };

    int s = 0;
    for (; s + kDepth <= steps; s += kDepth) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d) body(ring[d]);
    }
#pragma unroll
    for (int d = 0; d < kDepth - 1; ++d)
        if (s + d < steps) body(ring[d]);
    return viol;
}

// M > 1: groups of 8 R rows, R = rows_per_lane(MT).  Lane (rs, bs) takes the
// rows 8R g + rs + 8i (i < R) at beats bs, bs + 4, ...: each beat's code words
// are formed once per row and every activation word read from shared memory
// serves all R of the lane's rows.  Shared-memory reads of the activations
// were the bound with one row per lane (each dp4a of a lane consumed 4 / R
// bytes of them, against 128 bytes per clock per SM); two rows per lane with
// a deeper load ring measured faster than four.
// Weight rows per lane (2 or 4) per staged row count.  Measured on the 30-layer
// stack (ring depth per row in brackets): M = 2 121.1 us with four rows [2],
// 115.4 with two [4] (118.8 [3], 117.7 [5], 119.9 [6], 133.0 [8]; two rows at
// three CTAs per SM 127.6); M = 4 187.5 -> 183.6 (two rows [4], 2 classes);
// M = 8 311.6 -> 307.7 (two rows [2], 2 classes; [3] 325.2).
#ifndef TRIT_RPL_M2
#define TRIT_RPL_M2 2
#endif
#ifndef TRIT_RPL_M4
#define TRIT_RPL_M4 2
#endif
#ifndef TRIT_RPL_M8
#define TRIT_RPL_M8 2
#endif
__host__ __device__ constexpr int rows_per_lane(int mt) {
    return mt == 2 ? TRIT_RPL_M2 : mt == 4 ? TRIT_RPL_M4 : TRIT_RPL_M8;
}
__host__ __device__ constexpr int rows_per_group(int mt) { return 8 * rows_per_lane(mt); }

// Reduce-scatter of a lane's R x MT partial sums over the four lanes of its
// rows (lanes 4 rs + bs, bs = 0..3).  R = 4: after two butterfly steps lane bs
// holds the complete sums of its row i = 2 (bs & 1) + (bs >> 1) for every m
// (so the four lanes finish and store four different rows).  R = 2: lane bs
// holds those of row i = bs & 1 (lanes bs and bs ^ 2 hold the same row).
template <int MT, int R>
__device__ __forceinline__ void reduce_rows(const int (&acc)[R][MT], int bs, int (&out)[MT]) {
    const bool b0 = bs & 1, b1 = (bs >> 1) & 1;
    if constexpr (R == 2) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            const int send = b0 ? acc[0][m] : acc[1][m];
            const int t = (b0 ? acc[1][m] : acc[0][m]) + __shfl_xor_sync(~0u, send, 1);
            out[m] = t + __shfl_xor_sync(~0u, t, 2);
        }
        return;
    }
    constexpr int H = 2 * MT;   // values per half: rows {0, 1} or {2, 3}
    int t[H];
#pragma unroll
    for (int v = 0; v < H; ++v) {
        const int lo = acc[v / MT][v % MT], hi = acc[2 + v / MT][v % MT];
        const int send = b0 ? lo : hi;
        t[v] = (b0 ? hi : lo) + __shfl_xor_sync(~0u, send, 1);
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        const int send = b1 ? t[m] : t[MT + m];
        out[m] = (b1 ? t[MT + m] : t[m]) + __shfl_xor_sync(~0u, send, 2);
    }
}

// One beat of every row of a lane (M > 1): the two-bit code words of both
// 32-column halves of the lane's kRowsPerLane rows (v), multiplied by the MT
// staged activation rows of the beat at xp, added into acc.  With NJ weight
// classes the byte codes reach dp4a as (code word >> s) & (0x03030303 << 2k),
// byte value 4^k c, into accumulator k of NJ: NJ = 4 needs no shift (s = 0, k = j),
// NJ = 2 one shift by 4 for the upper two j (k = j & 1), NJ = 1 the shift by
// 2j (k = 0).  Accumulator k holds a multiple of 4^k; fold_classes divides it
// out exactly.  The caller may refill v's registers once this returns.
template <int MT, int NJ, int R>
__device__ __forceinline__ void mac_beat_rows(const uint4 (&v)[R], const uint4 *xp,
                                              int (&acc)[R][MT][NJ], uint32_t &viol) {
    static_assert(NJ == 1 || NJ == 2 || NJ == 4, "weight classes");
    uint32_t zw[2][R][2];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        viol |= (v[i].x & v[i].z) | (v[i].y & v[i].w);
        code_words(v[i].x, v[i].z, zw[0][i][0], zw[0][i][1]);
        code_words(v[i].y, v[i].w, zw[1][i][0], zw[1][i][1]);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            // activation words 4q..4q+3 of half h hold columns 8i + 4q + {0,1,2,3};
            // their codes are j = 2q (words 4q, 4q+1: even, odd code word) and
            // j = 2q + 1 (words 4q+2, 4q+3)
            constexpr uint32_t M0 = 0x03030303u;
            uint32_t c[R][4];
            int k0 = 0, k1 = 0;   // accumulator of the j = 2q / j = 2q + 1 codes
#pragma unroll
            for (int i = 0; i < R; ++i) {
                const uint32_t ze = zw[h][i][0], zo = zw[h][i][1];
                if (NJ == 4) {
                    c[i][0] = ze & (M0 << (4 * q));
                    c[i][1] = zo & (M0 << (4 * q));
                    c[i][2] = ze & (M0 << (4 * q + 2));
                    c[i][3] = zo & (M0 << (4 * q + 2));
                    k0 = 2 * q;
                    k1 = 2 * q + 1;
                } else if (NJ == 2) {
                    const uint32_t se = ze >> (4 * q), so = zo >> (4 * q);
                    c[i][0] = se & M0;
                    c[i][1] = so & M0;
                    c[i][2] = se & (M0 << 2);
                    c[i][3] = so & (M0 << 2);
                    k0 = 0;
                    k1 = 1;
                } else {
                    c[i][0] = (ze >> (4 * q)) & M0;
                    c[i][1] = (zo >> (4 * q)) & M0;
                    c[i][2] = (ze >> (4 * q + 2)) & M0;
                    c[i][3] = (zo >> (4 * q + 2)) & M0;
                    k0 = 0;
                    k1 = 0;
                }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const uint4 a = xp[4 * m + 2 * h + q];
#pragma unroll
                for (int i = 0; i < R; ++i) {
                    int t0 = acc[i][m][k0];
                    t0 = dp4a_su(a.x, c[i][0], t0);
                    t0 = dp4a_su(a.y, c[i][1], t0);
                    acc[i][m][k0] = t0;
                    int t1 = acc[i][m][k1];
                    t1 = dp4a_su(a.z, c[i][2], t1);
                    t1 = dp4a_su(a.w, c[i][3], t1);
                    acc[i][m][k1] = t1;
                }
            }
        }
    }
}

// sum_k acc[k] / 4^k, exact (accumulator k is a multiple of 4^k).
template <int NJ>
__device__ __forceinline__ int fold_classes(const int (&a)[NJ]) {
    int t = a[0];
#pragma unroll
    for (int k = 1; k < NJ; ++k) t += a[k] >> (2 * k);
    return t;
}

// Output m of row r of entry E from its complete integer sum v (column sum of
// the activation row already taken off).
__device__ __forceinline__ void store_out(const Entry &E, int m, int64_t r, int32_t v) {
    const int64_t o = int64_t(m) * E.N + r;
    if (E.acc) {
        atomicAdd(E.acc + o, v);
    } else {
        if (E.y_i32) E.y_i32[o] = v;
        if (E.y_f32) E.y_f32[o] = dequant(v, E.w_scale, E.x_scale[m]);
    }
}

// The M > 1 product loop over whole groups [gb, ge) of entry E: loads clamped
// to the planes (rows past N read row N - 1, beats past the row's end its last
// beat), D steps of loads in flight per row.
template <int MT, int D, int NJ>
__device__ __forceinline__ uint32_t run_groups_rows(const Entry &E, const uint32_t *xs,
                                                    const int32_t *s_xsum, int64_t gb,
                                                    int64_t ge, int rs, int bs) {
    constexpr int R = rows_per_lane(MT);
    constexpr int kRowsPerGroupM = rows_per_group(MT);
    constexpr int BV = beat_words(MT) / 4;   // uint4 per staged beat
    const int it = E.iters;
    const int steps = int(ge - gb) * it;
    const int64_t N = E.N;
    uint32_t viol = 0;

    // ---- load cursor
    const int last_beat = E.B - 1;
    const int64_t last_row = (ge * kRowsPerGroupM < N ? ge * kRowsPerGroupM : N) - 1;
    int64_t lrow = gb * kRowsPerGroupM + rs;
    auto row_at = [&](int64_t r) { return E.planes + (r < last_row ? r : last_row) * E.bstride; };
    const uint4 *lp[R];
#pragma unroll
    for (int i = 0; i < R; ++i) lp[i] = row_at(lrow + 8 * i);
    int lt = 0, loff = bs;
    auto next_load = [&](uint4 (&v)[R]) {
        const int o = loff < last_beat ? loff : last_beat;
#pragma unroll
        for (int i = 0; i < R; ++i) v[i] = ldg_stream(lp[i] + o);
        loff += kLanesPerRow;
        if (++lt == it) {
            lt = 0;
            loff = bs;
            lrow += kRowsPerGroupM;
#pragma unroll
            for (int i = 0; i < R; ++i) lp[i] = row_at(lrow + 8 * i);
        }
    };
    uint4 ring[D][R];
#pragma unroll
    for (int d = 0; d < D; ++d) next_load(ring[d]);

    int acc[R][MT][NJ];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int k = 0; k < NJ; ++k) acc[i][m][k] = 0;
    int64_t row = gb * kRowsPerGroupM + rs;
    int ct = 0;
    // this lane's staged beats: bs, bs + 4, ...; row m of a beat at 4m uint4
    const uint4 *xbase = reinterpret_cast<const uint4 *>(xs) + bs * BV;
    const uint4 *xp = xbase;

    auto body = [&](int slot) {
        uint4 v[R];
#pragma unroll
        for (int i = 0; i < R; ++i) v[i] = ring[slot][i];
        mac_beat_rows<MT, NJ, R>(v, xp, acc, viol);
        next_load(ring[slot]);
        xp += kLanesPerRow * BV;
        if (++ct == it) {
            // the row sums: each of the four lanes of a row group finishes one row
            int tot[R][MT];
#pragma unroll
            for (int i = 0; i < R; ++i)
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    tot[i][m] = fold_classes<NJ>(acc[i][m]);
#pragma unroll
                    for (int k = 0; k < NJ; ++k) acc[i][m][k] = 0;
                }
            int y[MT];
            reduce_rows<MT, R>(tot, bs, y);
            const int64_t r = row + 8 * (R == 4 ? 2 * (bs & 1) + (bs >> 1) : (bs & 1));
            if (r < N && (R == 4 || (bs >> 1) == 0)) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < rows_of(E)) store_out(E, m, r, y[m] - read_xsum_row<MT>(s_xsum, m));
            }
            ct = 0;
            xp = xbase;
            row += kRowsPerGroupM;
        }
    };

    int s = 0;
    for (; s + D <= steps; s += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) body(d);
    }
#pragma unroll
    for (int d = 0; d < D - 1; ++d)
        if (s + d < steps) body(d);
    return viol;
}

// M = 1 with rows of exactly 4*IT beats: the group loop is unrolled step by
// step, so every load, shared-memory read and accumulator index is static.
// The ring depth D divides IT, so step t of every group uses ring slot t % D;
// the last D loads of a group already fetch the next group's first beats.
// Optionally (kL2Ahead > 0) the group kL2Ahead further on (8 contiguous rows)
// is bulk-prefetched into L2 while a group is computed.

template <int IT>
__device__ __forceinline__ const uint4 *fixed_row_ptr(const Entry &E, int64_t g, int64_t last_row,
                                                      int rs) {
    const int64_t r = g * kRowsPerGroup + rs;
    return E.planes + (r < last_row ? r : last_row) * int64_t(E.bstride);
}

__device__ __forceinline__ int64_t fixed_last_row(const Entry &E, int64_t ge) {
    return (ge * kRowsPerGroup < E.N ? ge * kRowsPerGroup : E.N) - 1;
}

template <int IT, int D>
__device__ __forceinline__ uint32_t fixed_run(const Entry &E, const uint32_t *xs, float x_scale,
                                              int32_t xsum, int64_t gb, int64_t ge, int rs, int bs) {
    static_assert(IT % D == 0, "ring depth must divide the steps of a row");
    const int64_t N = E.N;
    int32_t *const y_i32 = E.y_i32;
    float *const y_f32 = E.y_f32;
    int32_t *const acc_out = E.acc;
    const float w_scale = E.w_scale;
    const int64_t last_row = fixed_last_row(E, ge);
    const uint4 *xb = reinterpret_cast<const uint4 *>(xs) + bs * kXBeatVec;
    // beat of step t: bs + kLanes1 t; only the last step can pass the row's end
    // (kLanes1 (IT - 1) < B <= kLanes1 IT), and there it is clamped to the row's
    // last beat, whose staged activations past B are zero
    const int last_off = bs + kLanes1 * (IT - 1) < E.B ? bs + kLanes1 * (IT - 1) : E.B - 1;
    auto off = [&](int t) { return t == IT - 1 ? last_off : bs + kLanes1 * t; };

    uint32_t viol = 0;
    const uint4 *rp = fixed_row_ptr<IT>(E, gb, last_row, rs);
    const uint4 *rpn = fixed_row_ptr<IT>(E, gb + 1, last_row, rs);
    uint4 ring[D];
#pragma unroll
    for (int d = 0; d < D; ++d) ring[d] = ldg_stream(rp + off(d));
    int64_t row = gb * kRowsPerGroup + rs;
    const bool pf = kL2Ahead > 0 && rs == 0 && bs == 0 && E.B == E.bstride;
    for (int64_t g = gb; g < ge; ++g) {
        if (pf && g + kL2Ahead < ge) {   // group g + kL2Ahead: 8 contiguous rows
            const int64_t r0 = (g + kL2Ahead) * kRowsPerGroup;
            const int64_t r1 = r0 + kRowsPerGroup < N ? r0 + kRowsPerGroup : N;
            if (r0 < r1)
                prefetch_l2_bulk(E.planes + r0 * E.bstride, uint32_t((r1 - r0) * E.bstride * 16));
        }
        int acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0;
#pragma unroll
        for (int t = 0; t < IT; ++t) {
            const uint4 v = ring[t % D];
            ring[t % D] = (t + D < IT) ? ldg_stream(rp + off(t + D))
                                       : ldg_stream(rpn + off(t + D - IT));
            viol |= (v.x & v.z) | (v.y & v.w);
            const uint4 *X = xb + t * (kLanes1 * kXBeatVec);
            const uint4 a0 = X[0], a1 = X[1], a2 = X[2], a3 = X[3];
            const uint32_t xl[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t xh[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
            mac_codes(v.x, v.z, xl, acc);
            mac_codes(v.y, v.w, xh, acc);
        }
        const int32_t y = row_sum1(codes_total(acc)) - xsum;
        if (bs == 0 && row < N) {
            if (acc_out) {
                atomicAdd(acc_out + row, y);
            } else {
                if (y_i32) y_i32[row] = y;
                if (y_f32) y_f32[row] = dequant(y, w_scale, x_scale);
            }
        }
        row += kRowsPerGroup;
        rp = rpn;
        rpn = fixed_row_ptr<IT>(E, g + 2, last_row, rs);
    }
    return viol;
}

template <int MT>
__global__ void __launch_bounds__(kThreads, min_blocks(MT))
    select_accumulate_kernel(const __grid_constant__ List L) {
    extern __shared__ __align__(16) uint32_t xs[];
    __shared__ int32_t s_xsum[kWarps];
    __shared__ float s_mlp_scale;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rs = lane / lanes_of(MT), bs = lane % lanes_of(MT);
    const int64_t lo = int64_t(blockIdx.x) * L.total_cost / gridDim.x;
    const int64_t hi = (int64_t(blockIdx.x) + 1) * L.total_cost / gridDim.x;
    uint32_t viol = 0;
    // A launch that follows on the stream with programmatic serialisation may
    // start its own set-up now (search, L2 prefetch of its first planes); every
    // CTA waits for the preceding grid (griddepcontrol.wait) before it reads
    // activations or writes anything.
    asm volatile("griddepcontrol.launch_dependents;");
    bool waited = false;

    int e = 0;   // last entry whose cost range starts at or before lo
    {
        int a = 0, b = L.count - 1;
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (L.e[mid].cost_begin <= lo) a = mid;
            else b = mid - 1;
        }
        e = a;
    }
    for (; e < L.count && L.e[e].cost_begin < hi; ++e) {
        const Entry &E = L.e[e];
        const int64_t gc = E.gcost;
        // groups whose first cost unit lies in [lo, hi)
        const int64_t dlo = lo - E.cost_begin, dhi = hi - E.cost_begin;
        const int64_t g0 = dlo <= 0 ? 0 : (dlo + gc - 1) / gc;
        int64_t g1 = (dhi + gc - 1) / gc;
        if (g1 > E.groups) g1 = E.groups;
        if (g0 >= g1) continue;
        const int64_t n = g1 - g0;
        const int64_t wb = g0 + n * warp / kWarps, we = g0 + n * (warp + 1) / kWarps;
        // 1: rows of 40 beats, 2: rows of 108 beats (unrolled paths), 0: generic
        const int path = (MT == 1 && E.B == 40 && E.iters == kIt40) ? 1
                       : (MT == 1 && E.B == 108 && E.iters == kIt108) ? 2 : 0;
        // start this warp's first groups streaming into L2 before the barrier
        constexpr int kRows = MT == 1 ? kRowsPerGroup : rows_per_group(MT);
        if (TRIT_PREFETCH_FIRST && lane == 0 && wb < we && E.B == E.bstride) {
            const int64_t r0 = wb * kRows;
            const int64_t ahead = TRIT_PREFETCH_FIRST;
            int64_t r1 = (wb + ahead < we ? wb + ahead : we) * kRows;
            r1 = r1 < E.N ? r1 : E.N;
            prefetch_l2_bulk(E.planes + r0 * E.bstride, uint32_t((r1 - r0) * E.bstride * 16));
        }
        __syncthreads();   // the previous entry's readers are done with xs
        if (!waited) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            waited = true;
        }
        float xsc;
        if (MT == 1 && mlp_of(E)) {
            stage_x_intmlp(E, L.mlp[mlp_of(E) - 1], xs, g0 == 0, s_xsum, &s_mlp_scale);
            xsc = 0.0f;   // read from s_mlp_scale after the barrier
        } else if (MT == 1 && E.xf) {
            xsc = stage_x_fp32(E, xs, g0 == 0, L.err, s_xsum);
        } else {
            stage_x<MT>(E, xs, s_xsum);
            xsc = E.x_scale ? E.x_scale[0] : L.x_scale_val;
        }
        __syncthreads();
        const int32_t xsum = MT == 1 ? read_xsum(s_xsum) : 0;
        if (MT == 1 && mlp_of(E)) xsc = s_mlp_scale;
        if (wb < we) {
            if constexpr (MT == 1) {
                if (path == 1)
                    viol |= fixed_run<kIt40, TRIT_RING_40>(E, xs, xsc, xsum, wb, we, rs, bs);
                else if (path == 2)
                    viol |= fixed_run<kIt108, TRIT_RING_108>(E, xs, xsc, xsum, wb, we, rs, bs);
                else
                    viol |= run_groups(E, xs, xsc, xsum, wb, we, rs, bs);
            } else {
                viol |= run_groups_rows<MT, ring_rows(MT), acc_classes(MT)>(E, xs, s_xsum, wb, we, rs, bs);
            }
        }
    }
    if (__any_sync(~0u, viol != 0) && lane == 0) atomicOr(L.err, TRIT_ERR_P1);
}


// Small M = 1 launches, every warp one group at most (the per-matvec launches
// of a dependency-ordered token).  Each lane copies all of its group's beats
// into shared memory at once (cp.async), so the product waits for one memory
// round trip, not one per ring refill.  Where every entry's planes are marked
// ready (complete before the preceding kernel was launched) the copies start as
// soon as the CTA is resident -- under programmatic serialisation while the
// preceding grid still runs -- and after griddepcontrol.wait only the staging
// of the activations and the products out of shared memory remain; otherwise
// they start after the wait.
//
// Groups are numbered across the list (Entry.cost_begin: the entry's first
// group; the list's total_cost: all groups); warp w of CTA b takes group
// 8b + w, or (split lists, flags bit 2, when twice the CTAs fit one wave)
// warps w and w + 4 take group 4b + w, one half of its steps each, the second
// half's code sums joining the first's through shared memory.  Shared memory:
// the staged activations (xs_words), then per warp plane_steps x 32 lanes x
// 16 bytes of planes, lane-interleaved so each step's reads are contiguous,
// then (IntMlp rows) the row's signed fp32 products.
//
// Paired lists (flags bit 1: the gate and up projections of IntMlp blocks,
// entries 2p and 2p + 1, one input row): the c-th CTA of pair p stages the row
// once, its warps 0-3 take gate groups 4c..4c+3 and warps 4-7 the same up
// groups, and after the products warp 0 forms t = relu(a_gate)^2 a_up of the
// CTA's 32 rows and publishes their max |t| as partial c of the pair's
// descriptor ("Tritium ..." -- Numerics, IntMlp).  An entry with an IntMlp
// descriptor in an unpaired list stages its row from those partials
// (stage_x_intmlp_parts).
__global__ void __launch_bounds__(kThreads, 2) select_accumulate_pre_kernel(const __grid_constant__ List L) {
    static_assert(kWarps == 8, "paired and split lists divide the CTA into two halves of four warps");
    extern __shared__ __align__(16) uint32_t xs[];
    __shared__ int32_t s_xsum[kWarps];
    __shared__ float s_mlp_scale;
    __shared__ int32_t s_pair[2][4][kRowsPerGroup];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rs = lane / kLanes1, bs = lane % kLanes1;
    asm volatile("griddepcontrol.launch_dependents;");
    uint4 *pl = reinterpret_cast<uint4 *>(xs + L.xs_words) + (warp * L.plane_steps) * 32 + lane;
    const int64_t G = L.total_cost;
    const bool paired = (L.flags & 2) != 0;
    const bool split = (L.flags & 4) != 0;   // two warps per group, one per half of the row
    const int half = split ? warp >> 2 : 0;
    const int64_t cta0 = int64_t(blockIdx.x) * (split ? 4 : kWarps);
    auto entry_of = [&](int64_t gw) {   // last entry whose first group is <= gw
        int a = 0, b = L.count - 1;
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (L.e[mid].cost_begin <= gw) a = mid;
            else b = mid - 1;
        }
        return a;
    };
    // this warp's entry (-1: none) and group, and the entries the CTA stages
    int we = -1, e0, e1;
    int64_t g = 0, pc = 0;
    if (paired) {   // gate and up share cost_begin, so the search lands on up
        const int eu = entry_of(cta0), eg = eu - 1;
        pc = int64_t(blockIdx.x) - L.e[eg].cost_begin / kWarps;
        g = 4 * pc + (warp & 3);
        const int ew = warp < 4 ? eg : eu;
        we = g < L.e[ew].groups ? ew : -1;
        e0 = e1 = eg;
    } else {
        const int span = split ? 4 : kWarps;
        const int64_t gw = cta0 + (split ? (warp & 3) : warp);
        if (gw < G) {
            we = entry_of(gw);
            g = gw - L.e[we].cost_begin;
        }
        const int64_t last = cta0 + span - 1 < G ? cta0 + span - 1 : G - 1;
        e0 = entry_of(cta0);
        e1 = entry_of(last);
    }
    // this warp's steps [t0, t1) of its group's rows (split: one half each)
    int t0 = 0, t1 = 0;
    if (we >= 0) {
        const int it = L.e[we].iters, ith = (it + 1) / 2;
        t0 = split ? half * ith : 0;
        t1 = split ? (t0 + ith < it ? t0 + ith : it) : it;
    }
    auto copy_planes = [&]() {
        if (we < 0) return;
        const Entry &E = L.e[we];
        const int64_t r = g * kRowsPerGroup + rs;
        const uint4 *rp = E.planes + (r < E.N ? r : E.N - 1) * int64_t(E.bstride);
        // beat of step t: bs + 4t, clamped to the row's last beat (the staged
        // activations past the row's end are zero)
        for (int t = t0; t < t1; ++t) {
            const int beat = bs + kLanes1 * t;
            cpa16(pl + (t - t0) * 32, rp + (beat < E.B ? beat : E.B - 1));
        }
        cpa_commit();
    };
    // planes written by the preceding kernel are visible only after the wait
    const bool early = (L.flags & 1) != 0;
    if (early) copy_planes();
    uint32_t viol = 0;
    int32_t my_part = 0, my_xsum = 0;   // this lane's row code sum and the staged row's column sum
    float my_xsc = 0.0f;
    for (int e = e0; e <= e1; ++e) {
        const Entry &E = L.e[e];
        if (e == e0) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            if (!early) copy_planes();
        } else {
            __syncthreads();   // the previous entry's readers are done with xs
        }
        // the CTA that holds the entry's group 0 writes its codes and scale
        const bool owner = paired ? pc == 0 : E.cost_begin >= cta0;
        const bool intmlp = !paired && mlp_of(E) != 0;
        float xsc;
        if (intmlp) {
            stage_x_intmlp_parts(E, L.mlp[mlp_of(E) - 1], xs,
                                 reinterpret_cast<int32_t *>(xs + L.xs_words) +
                                     kWarps * L.plane_steps * 128,
                                 owner, s_xsum, &s_mlp_scale);
            xsc = 0.0f;   // read from s_mlp_scale after the barrier
        } else if (E.xf) {
            xsc = stage_x_fp32(E, xs, owner, L.err, s_xsum);
        } else {
            stage_x<1>(E, xs, s_xsum);
            xsc = E.x_scale ? E.x_scale[0] : L.x_scale_val;
        }
        __syncthreads();
        const int32_t xsum = read_xsum(s_xsum);
        if (intmlp) xsc = s_mlp_scale;
        if (we < 0 || (!paired && we != e)) continue;
        cpa_wait_all();
        const uint4 *xb = reinterpret_cast<const uint4 *>(xs) + bs * kXBeatVec;
        int acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0;
#pragma unroll 2
        for (int t = t0; t < t1; ++t) {
            const uint4 v = pl[(t - t0) * 32];
            viol |= (v.x & v.z) | (v.y & v.w);
            const uint4 *X = xb + t * (kLanes1 * kXBeatVec);
            const uint4 a0 = X[0], a1 = X[1], a2 = X[2], a3 = X[3];
            const uint32_t xl[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const uint32_t xh[8] = {a2.x, a2.y, a2.z, a2.w, a3.x, a3.y, a3.z, a3.w};
            mac_codes(v.x, v.z, xl, acc);
            mac_codes(v.y, v.w, xh, acc);
        }
        my_part = row_sum1(codes_total(acc));
        my_xsum = xsum;
        my_xsc = xsc;
    }
    int32_t y = my_part - my_xsum;
    if (split) {   // the second half's code sums join the first half's (same rows)
        if (half == 1 && bs == 0) s_pair[0][warp & 3][rs] = my_part;
        __syncthreads();
        y += s_pair[0][warp & 3][rs];
    }
    const int64_t row = g * kRowsPerGroup + rs;
    const bool mine = we >= 0 && half == 0 && row < L.e[we].N;
    if (mine && bs == 0) {
        const Entry &W = L.e[we];   // paired: the up warps' entry is not the staged one
        if (W.acc) {
            atomicAdd(W.acc + row, y);
        } else {
            if (W.y_i32) W.y_i32[row] = y;
            if (W.y_f32) W.y_f32[row] = dequant(y, W.w_scale, my_xsc);
        }
    }
    if (paired) {
        if (bs == 0) s_pair[warp >> 2][warp & 3][rs] = mine ? y : 0;
        __syncthreads();
        if (warp == 0) {
            bool neg;
            const trit_u128 t = intmlp_abs_t(s_pair[0][lane >> 3][lane & 7],
                                             s_pair[1][lane >> 3][lane & 7], neg);
            uint64_t hi = uint64_t(t >> 64), lo = uint64_t(t);
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                const uint64_t h2 = __shfl_xor_sync(~0u, hi, o), l2 = __shfl_xor_sync(~0u, lo, o);
                if (h2 > hi || (h2 == hi && l2 > lo)) {
                    hi = h2;
                    lo = l2;
                }
            }
            const MlpDesc &D = L.mlp[mlp_of(L.e[e0]) - 1];
            if (lane == 0) {
                D.tmax[2 * pc] = hi;
                D.tmax[2 * pc + 1] = lo;
            }
            // each row's signed fp32 product, for the down launch's codes
            mlp_tf_of(D.tmax, D.ntmax)[32 * pc + lane] =
                intmlp_tf(s_pair[0][lane >> 3][lane & 7], s_pair[1][lane >> 3][lane & 7]);
        }
    }
    if (__any_sync(~0u, viol != 0) && lane == 0) atomicOr(L.err, TRIT_ERR_P1);
}

// Shared memory a pre-loading launch may take (the staged activations and
// every warp's planes); larger lists take the streaming kernel.  TRIT_PRE_LOAD
// 0 keeps small lists on the streaming kernel (the MLP block calls still use
// the pre-loading one).
constexpr size_t kPreSmemMax = 225 * 1024;
#ifndef TRIT_PRE_LOAD
#define TRIT_PRE_LOAD 1
#endif
#ifndef TRIT_PRE_SPLIT
#define TRIT_PRE_SPLIT 1
#endif

__host__ __device__ constexpr int64_t pre_iters(int64_t K) { return ((K + 63) / 64 + kLanes1 - 1) / kLanes1; }
// Shared memory of a pre-loading launch whose longest row has `iters` steps:
// the staged activations, every warp's planes and, with IntMlp rows, two
// arrays of iters x 256 words: the staging uses one (the signed fp32
// products); the size also keeps one such CTA per SM (measured: two sharing
// an SM made the ordered token 7% slower).
size_t pre_smem(int64_t iters, bool intmlp = false) {
    return size_t(iters) * kLanes1 * kXBeatWords * 4 + size_t(kWarps) * iters * 32 * 16 +
           (intmlp ? size_t(iters) * 2 * 256 * 4 : 0);
}

// Launch entries[0..n) (M = 1) on the pre-loading kernel when every entry
// holds whole rows and, unless forced, the list's groups fit one resident wave
// with one group per warp.  Returns false (nothing launched) otherwise; true
// with the launch's status in `status`.  Paired lists: entries 2p, 2p + 1 are
// the gate and up products of IntMlp block p (mlp[p] receives the partials).
// Resident CTAs per SM of the pre-loading kernel with `smem` bytes of dynamic
// shared memory (a few sizes recur: cached).  The first call on a device sets
// the kernel's shared-memory limit and carve-out.
cudaError_t pre_occupancy(size_t smem, int &occ) {
    struct Slot { int dev; size_t smem; int occ; };
    static thread_local Slot cache[8];
    static thread_local int used = 0, next = 0, ready_dev = -1;
    int dev = 0;
    cudaError_t st = cudaGetDevice(&dev);
    if (st != cudaSuccess) return st;
    for (int i = 0; i < used; ++i)
        if (cache[i].dev == dev && cache[i].smem == smem) {
            occ = cache[i].occ;
            return cudaSuccess;
        }
    if (ready_dev != dev) {
        st = cudaFuncSetAttribute(select_accumulate_pre_kernel,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, int(kPreSmemMax));
        if (st != cudaSuccess) return st;
        // one shared-memory carve-out for every launch of this kernel, so that
        // the CTAs of a launch can become resident beside those of the one
        // before it (a carve-out change waits for the SM to drain)
        st = cudaFuncSetAttribute(select_accumulate_pre_kernel,
                                  cudaFuncAttributePreferredSharedMemoryCarveout,
                                  int(cudaSharedmemCarveoutMaxShared));
        if (st != cudaSuccess) return st;
        ready_dev = dev;
    }
    st = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, select_accumulate_pre_kernel, kThreads,
                                                       smem);
    if (st != cudaSuccess) return st;
    cache[next] = Slot{dev, smem, occ};
    next = (next + 1) % 8;
    if (used < 8) ++used;
    return cudaSuccess;
}

// Launch entries[0..n) (M = 1) on the pre-loading kernel when every entry
// holds whole rows and, unless forced, the list's groups fit one resident wave
// with one group per warp.  Returns false (nothing launched) otherwise; true
// with the launch's status in `status`.  Paired lists: entries 2p, 2p + 1 are
// the gate and up products of IntMlp block p (mlp[p] receives the partials).
// Unpaired lists take two warps per group (split) when twice the CTAs, each
// holding half the steps' planes, still fit one wave.
bool launch_list_pre(const Entry *entries, int n, uint32_t *err, cudaStream_t s,
                     float x_scale_val, cudaError_t &status, const MlpDesc *mlp = nullptr,
                     int nmlp = 0, bool paired = false, bool force = false) {
    if (!force && !TRIT_PRE_LOAD) return false;
    int64_t groups = 0, grid = 0;
    int max_iters = 1;
    bool early = true;
    if (paired && n % 2) return false;
    for (int i = 0; i < n; ++i) {
        if (entries[i].B != entries[i].bstride || rows_of(entries[i]) != 1) return false;
        early = early && (entries[i].mrows & kPlanesReady) != 0;
        groups += entries[i].groups;
        if (entries[i].iters > max_iters) max_iters = entries[i].iters;
    }
    const int xs_words = max_iters * kLanes1 * kXBeatWords;
    const bool rows = nmlp > 0 && !paired;   // IntMlp rows staged through shared memory
    auto smem_of = [&](int steps) {
        return size_t(xs_words) * 4 + size_t(kWarps) * steps * 32 * 16 +
               (rows ? size_t(max_iters) * 2 * 256 * 4 : 0);
    };
    const int64_t sms = device_sm_count();
    int steps = max_iters, occ = 0;
    bool split = false;
    if (!paired && TRIT_PRE_SPLIT && smem_of((max_iters + 1) / 2) <= kPreSmemMax) {
        status = pre_occupancy(smem_of((max_iters + 1) / 2), occ);
        if (status != cudaSuccess) return true;
        if ((groups + 3) / 4 <= int64_t(occ) * sms) {
            split = true;
            steps = (max_iters + 1) / 2;
            grid = (groups + 3) / 4;
        }
    }
    const size_t smem = smem_of(steps);
    if (smem > kPreSmemMax) return false;
    if (!split) {
        status = pre_occupancy(smem, occ);
        if (status != cudaSuccess) return true;
    }
    // lists longer than a wave go to the streaming kernel: decided before any
    // copying (a decode step's list takes this exit on every launch)
    if (!force && !paired && !split && (groups + kWarps - 1) / kWarps > int64_t(occ) * sms)
        return false;
    static thread_local List L;
    if (paired) {
        for (int p = 0; p < n / 2; ++p) {
            L.e[2 * p] = entries[2 * p];
            L.e[2 * p + 1] = entries[2 * p + 1];
            L.e[2 * p].cost_begin = L.e[2 * p + 1].cost_begin = grid * kWarps;
            grid += (entries[2 * p].groups + 3) / 4;
        }
    } else {
        int64_t g = 0;
        for (int i = 0; i < n; ++i) {
            L.e[i] = entries[i];
            L.e[i].cost_begin = g;
            g += entries[i].groups;
        }
        if (!split) grid = (groups + kWarps - 1) / kWarps;
    }
    if (!force && grid > int64_t(occ) * sms) return false;
    L.count = n;
    L.err = err;
    L.x_scale_val = x_scale_val;
    L.flags = (early ? 1 : 0) | (paired ? 2 : 0) | (split ? 4 : 0);
    L.plane_steps = steps;
    for (int i = 0; i < kMaxMlp; ++i) L.mlp[i] = i < nmlp ? mlp[i] : MlpDesc{};
    L.total_cost = paired ? grid * kWarps : groups;
    L.xs_words = xs_words;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    status = cudaLaunchKernelEx(&cfg, select_accumulate_pre_kernel, L);
    return true;
}

template <int MT>
int occupancy(size_t smem) {
    // cached per (shared-memory size, device); sizes repeat from call to call
    static thread_local size_t last_smem = ~size_t(0);
    static thread_local int last_dev = -1, last_occ = 1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (smem != last_smem || dev != last_dev) {
        int occ = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, select_accumulate_kernel<MT>, kThreads,
                                                      smem);
        last_occ = occ < 1 ? 1 : occ;
        last_smem = smem;
        last_dev = dev;
    }
    return last_occ;
}

template <int MT>
cudaError_t launch_list(const Entry *entries, int n, uint32_t *err, cudaStream_t s,
                        const MlpDesc *mlp = nullptr, int nmlp = 0, float x_scale_val = 0.0f) {
    if (MT == 1 && nmlp == 0) {
        cudaError_t st = cudaSuccess;
        if (launch_list_pre(entries, n, err, s, x_scale_val, st)) return st;
    }
    static thread_local List L;   // host staging for the by-value parameter block
    L.count = n;
    L.err = err;
    L.x_scale_val = x_scale_val;
    L.flags = 0;
    L.plane_steps = 0;
    L.pad_ = 0;
    for (int i = 0; i < kMaxMlp; ++i) L.mlp[i] = i < nmlp ? mlp[i] : MlpDesc{};
    int64_t cost = 0, groups = 0;
    int max_iters = 1;
    for (int i = 0; i < n; ++i) {
        L.e[i] = entries[i];
        cost += stage_cost(MT);   // staging the entry's rows, charged to whoever starts it
        L.e[i].cost_begin = cost;
        cost += entries[i].groups * entries[i].gcost;
        groups += entries[i].groups;
        if (entries[i].iters > max_iters) max_iters = entries[i].iters;
    }
    L.total_cost = cost;
    L.xs_words = max_iters * lanes_of(MT) * beat_words(MT);
    const size_t smem = size_t(L.xs_words) * 4;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(select_accumulate_kernel<MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(smem));
        if (e != cudaSuccess) return e;
    }
    const int64_t cap = int64_t(occupancy<MT>(smem)) * device_sm_count() * TRIT_WAVES;
    const int64_t want = (groups + kWarps - 1) / kWarps;
    const int grid = int(want < cap ? (want < 1 ? 1 : want) : cap);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, select_accumulate_kernel<MT>, L);
}

// The fp32 pass of segmented products: y_f32 = dequant(acc) where acc is the
// product's int32 sums (y_i32, or the y_f32 buffer itself read as int32).
__global__ void __launch_bounds__(256) segment_epilogue_kernel(const int32_t *acc, float *y_f32,
                                                               int64_t M, int64_t N, float w_scale,
                                                               const float *x_scale,
                                                               float x_scale_val) {
    const int64_t total = M * N;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t m = i / N;
        y_f32[i] = dequant(acc[i], w_scale, x_scale ? x_scale[m] : x_scale_val);
    }
}

// One list entry: activation rows [m0, m0 + mrows) and beats [b0, b0 + nb) of p.
Entry make_entry(const ProjDev &p, int64_t m0, int mrows, int64_t b0, int64_t nb, int32_t *acc,
                 int lanes) {
    Entry E;
    const int64_t Kp = int64_t(p.B) * 64;
    E.planes = p.planes + b0;
    E.x = p.x ? p.x + m0 * Kp + b0 * 64 : nullptr;
    E.xf = p.xf;                 // fused entries are single-segment, M = 1
    E.x_i8_out = p.x_i8_out;
    E.x_scale = p.x_scale ? p.x_scale + m0 : nullptr;
    E.y_i32 = p.y_i32 ? p.y_i32 + m0 * p.N : nullptr;
    E.y_f32 = p.y_f32 ? p.y_f32 + m0 * p.N : nullptr;
    E.acc = acc ? acc + m0 * p.N : nullptr;
    E.N = p.N;
    E.groups = (p.N + kRowsPerGroup - 1) / kRowsPerGroup;
    E.cost_begin = 0;
    E.xld = int32_t(Kp);
    const int64_t kseg = int64_t(p.K) - b0 * 64;
    E.K = int32_t(kseg < nb * 64 ? kseg : nb * 64);
    E.B = int32_t(nb);
    E.iters = int32_t((nb + lanes - 1) / lanes);
    E.bstride = p.B;
    E.mrows = mrows | (p.planes_ready ? kPlanesReady : 0);
    E.gcost = E.iters * (nb == 108 ? TRIT_COST_108 : 100);
    E.w_scale = p.w_scale;
    return E;
}

template <int MT>
cudaError_t launch_entries(const Entry *all, int count, uint32_t *err, cudaStream_t s,
                           float x_scale_val) {
    for (int base = 0; base < count; base += kMaxList) {
        const int n = count - base < kMaxList ? count - base : kMaxList;
        cudaError_t e = launch_list<MT>(all + base, n, err, s, nullptr, 0, x_scale_val);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Expand the products into list entries -- activation rows MT at a time, and
// column segments for rows longer than seg_beats(MT) -- and launch them.  A
// product whose x_scale is NULL (M = 1) takes x_scale_val as its input scale;
// such a product is launched on its own (count == 1).
template <int MT>
cudaError_t launch_products(const ProjDev *list, int count, uint32_t *err, cudaStream_t s) {
    static thread_local Entry buf[kMaxList];
    int n = 0;
    cudaError_t e = cudaSuccess;
    float xs_val = 0.0f;
    for (int i = 0; i < count; ++i)
        if (!list[i].x_scale && !list[i].xf) {
            if (count != 1 || MT != 1 || list[i].M != 1) return cudaErrorInvalidValue;
            xs_val = list[i].x_scale_val;
        }
    // zero the accumulation targets of segmented products first
    for (int i = 0; i < count && e == cudaSuccess; ++i) {
        const ProjDev &p = list[i];
        if (p.B > seg_beats(MT)) {
            int32_t *acc = p.y_i32 ? p.y_i32 : reinterpret_cast<int32_t *>(p.y_f32);
            e = cudaMemsetAsync(acc, 0, size_t(p.M * p.N) * sizeof(int32_t), s);
        }
    }
    for (int i = 0; i < count && e == cudaSuccess; ++i) {
        const ProjDev &p = list[i];
        const bool seg = p.B > seg_beats(MT);
        int32_t *acc = !seg ? nullptr : (p.y_i32 ? p.y_i32 : reinterpret_cast<int32_t *>(p.y_f32));
        for (int64_t m0 = 0; m0 < p.M && e == cudaSuccess; m0 += MT) {
            const int rows = int(p.M - m0 < MT ? p.M - m0 : MT);
            for (int64_t b0 = 0; b0 < p.B && e == cudaSuccess; b0 += seg_beats(MT)) {
                const int64_t nb = p.B - b0 < seg_beats(MT) ? p.B - b0 : seg_beats(MT);
                buf[n] = make_entry(p, m0, rows, b0, nb, acc, lanes_of(MT));
                if (MT > 1) buf[n].groups = (p.N + rows_per_group(MT) - 1) / rows_per_group(MT);
                ++n;
                if (n == kMaxList) {
                    e = launch_entries<MT>(buf, n, err, s, xs_val);
                    n = 0;
                }
            }
        }
    }
    if (e == cudaSuccess && n) e = launch_entries<MT>(buf, n, err, s, xs_val);
    for (int i = 0; i < count && e == cudaSuccess; ++i) {
        const ProjDev &p = list[i];
        if (p.B > seg_beats(MT) && p.y_f32) {
            const int32_t *acc = p.y_i32 ? p.y_i32 : reinterpret_cast<const int32_t *>(p.y_f32);
            const int64_t total = p.M * p.N;
            int64_t blocks = (total + 255) / 256;
            const int64_t cap = int64_t(device_sm_count()) * 8;
            blocks = blocks < cap ? blocks : cap;
            segment_epilogue_kernel<<<int(blocks), 256, 0, s>>>(acc, p.y_f32, p.M, p.N, p.w_scale,
                                                                p.x_scale, p.x_scale_val);
            e = cudaGetLastError();
        }
    }
    return e;
}

}  // namespace

cudaError_t launch_gemv_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s) {
    return launch_products<1>(list, count, err, s);
}

// IntMlp down projections: up to kMaxMlp per launch (each entry single-segment,
// its row staged from the gate and up outputs).
cudaError_t launch_intmlp_gemv_many(const MlpProjDev *list, int count, uint32_t *err,
                                    cudaStream_t s) {
    static thread_local Entry buf[kMaxMlp];
    static thread_local MlpDesc desc[kMaxMlp];
    for (int base = 0; base < count; base += kMaxMlp) {
        const int n = count - base < kMaxMlp ? count - base : kMaxMlp;
        for (int i = 0; i < n; ++i) {
            const MlpProjDev &m = list[base + i];
            buf[i] = make_entry(m.down, 0, 1, 0, m.down.B, nullptr, kLanes1);
            buf[i].mrows |= (i + 1) << 8;
            desc[i].a_gate = m.a_gate;
            desc[i].a_up = m.a_up;
            desc[i].x_scale = m.x_scale_in;
            desc[i].w_gate = m.w_gate;
            desc[i].w_up = m.w_up;
            desc[i].tmax = nullptr;
            desc[i].ntmax = 0;
            desc[i].pad_ = 0;
        }
        cudaError_t e = launch_list<1>(buf, n, err, s, desc, n);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// ---- batch-1 MLP blocks in two launches ------------------------------------------

int64_t mlp_tmax_parts(int64_t F) { return ((F + kRowsPerGroup - 1) / kRowsPerGroup + 3) / 4; }

bool mlp_pairs_supported(int64_t K, int64_t F) {
    return pre_smem(pre_iters(K)) <= kPreSmemMax && pre_smem(pre_iters(F), true) <= kPreSmemMax;
}

// Gate and up of each block.  Blocks that the pre-loading kernel takes go as
// paired lists (publishing the max|t| partials) when all their 32-row tiles
// fit one resident wave -- the batch-1 chain of one block per call; longer
// lists go as fused quantise-and-multiply products on the streaming kernel,
// followed by one launch forming the same partials from a_gate and a_up.
// Blocks the pre-loading kernel does not take need no partials (their down
// launch reduces max|t| itself).
cudaError_t launch_mlp_gate_up(const MlpBlockDev *list, int count, uint32_t *err, cudaStream_t s) {
    static thread_local Entry buf[2 * kMaxMlp];
    static thread_local MlpDesc desc[kMaxMlp];
    static thread_local ProjDev rest[TRIT_MAX_LIST_PER_LAUNCH];
    static thread_local MlpTmaxJob jobs[TRIT_MAX_LIST_PER_LAUNCH];
    int n = 0, nr = 0, nj = 0;
    cudaError_t e = cudaSuccess;
    int64_t tiles = 0;
    int iters = 1;
    for (int i = 0; i < count; ++i)
        if (mlp_pairs_supported(list[i].gate.K, list[i].gate.N)) {
            tiles += mlp_tmax_parts(list[i].gate.N);
            const int it = int(pre_iters(list[i].gate.K));
            iters = it > iters ? it : iters;
        }
    bool paired = true;
    if (tiles) {
        int occ = 0;
        e = pre_occupancy(pre_smem(iters), occ);
        if (e != cudaSuccess) return e;
        paired = tiles <= int64_t(occ) * device_sm_count();
    }
    if (!paired) {
        for (int i = 0; i < count && e == cudaSuccess; ++i) {
            const MlpBlockDev &b = list[i];
            rest[nr++] = b.gate;
            rest[nr++] = b.up;
            if (mlp_pairs_supported(b.gate.K, b.gate.N))
                jobs[nj++] = MlpTmaxJob{b.gate.y_i32, b.up.y_i32, b.gate.N, b.tmax};
            if (nr + 2 > TRIT_MAX_LIST_PER_LAUNCH) {
                e = launch_gemv_many(rest, nr, err, s);
                if (e == cudaSuccess && nj) e = launch_mlp_tmax(jobs, nj, s);
                nr = nj = 0;
            }
        }
        if (e == cudaSuccess && nr) e = launch_gemv_many(rest, nr, err, s);
        if (e == cudaSuccess && nj) e = launch_mlp_tmax(jobs, nj, s);
        return e;
    }
    auto flush = [&]() {
        if (n && e == cudaSuccess &&
            !launch_list_pre(buf, 2 * n, err, s, 0.0f, e, desc, n, true, true))
            e = cudaErrorInvalidValue;
        n = 0;
    };
    auto flush_rest = [&]() {
        if (nr && e == cudaSuccess) e = launch_gemv_many(rest, nr, err, s);
        nr = 0;
    };
    for (int i = 0; i < count && e == cudaSuccess; ++i) {
        const MlpBlockDev &b = list[i];
        if (mlp_pairs_supported(b.gate.K, b.gate.N)) {
            buf[2 * n] = make_entry(b.gate, 0, 1, 0, b.gate.B, nullptr, kLanes1);
            buf[2 * n].mrows |= (n + 1) << 8;
            buf[2 * n + 1] = make_entry(b.up, 0, 1, 0, b.up.B, nullptr, kLanes1);
            desc[n] = MlpDesc{};
            desc[n].tmax = b.tmax;
            desc[n].ntmax = int32_t(mlp_tmax_parts(b.gate.N));
            if (++n == kMaxMlp) flush();
        } else {
            rest[nr++] = b.gate;
            rest[nr++] = b.up;
            if (nr + 2 > TRIT_MAX_LIST_PER_LAUNCH) flush_rest();
        }
    }
    flush();
    flush_rest();
    return e;
}

// The down projection of each block, its row formed from the gate and up
// outputs: from the published partials on the pre-loading kernel, else by the
// streaming kernel's own max|t| pass.
cudaError_t launch_mlp_down(const MlpBlockDev *list, int count, uint32_t *err, cudaStream_t s) {
    static thread_local Entry buf[kMaxMlp];
    static thread_local MlpDesc desc[kMaxMlp];
    static thread_local MlpProjDev rest[kMaxMlp];
    int n = 0, nr = 0;
    cudaError_t e = cudaSuccess;
    auto flush = [&]() {
        if (n && e == cudaSuccess && !launch_list_pre(buf, n, err, s, 0.0f, e, desc, n, false, true))
            e = cudaErrorInvalidValue;
        n = 0;
    };
    auto flush_rest = [&]() {
        if (nr && e == cudaSuccess) e = launch_intmlp_gemv_many(rest, nr, err, s);
        nr = 0;
    };
    for (int i = 0; i < count && e == cudaSuccess; ++i) {
        const MlpBlockDev &b = list[i];
        if (mlp_pairs_supported(b.gate.K, b.gate.N)) {
            buf[n] = make_entry(b.down, 0, 1, 0, b.down.B, nullptr, kLanes1);
            buf[n].mrows |= (n + 1) << 8;
            desc[n].a_gate = b.gate.y_i32;
            desc[n].a_up = b.up.y_i32;
            desc[n].x_scale = b.gate.x_scale;
            desc[n].w_gate = b.w_gate;
            desc[n].w_up = b.w_up;
            desc[n].tmax = b.tmax;
            desc[n].ntmax = int32_t(mlp_tmax_parts(b.gate.N));
            desc[n].pad_ = 0;
            if (++n == kMaxMlp) flush();
        } else {
            MlpProjDev &m = rest[nr++];
            m.down = b.down;
            m.a_gate = b.gate.y_i32;
            m.a_up = b.up.y_i32;
            m.x_scale_in = b.gate.x_scale;
            m.w_gate = b.w_gate;
            m.w_up = b.w_up;
            if (nr == kMaxMlp) flush_rest();
        }
    }
    flush();
    flush_rest();
    return e;
}

// Activation rows are taken 8 at a time; a product's remaining r < 8 rows go
// to the kernel staging 2 (r <= 2), 4 (r <= 4) or 8 rows, so no chunk stages
// more empty rows than it must.  Every chunk re-reads the planes.
cudaError_t launch_gemm_dp4a_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s) {
    static thread_local ProjDev by8[TRIT_MAX_LIST_PER_LAUNCH], by4[TRIT_MAX_LIST_PER_LAUNCH],
        by2[TRIT_MAX_LIST_PER_LAUNCH];
    int n8 = 0, n4 = 0, n2 = 0;
    for (int i = 0; i < count; ++i) {
        const ProjDev &p = list[i];
        const int64_t full = p.M / 8 * 8, r = p.M - full;
        if (full) {
            by8[n8] = p;
            by8[n8++].M = full;
        }
        if (r) {
            ProjDev q = p;
            const int64_t Kp = int64_t(p.B) * 64;
            q.x = p.x ? p.x + full * Kp : nullptr;
            q.x_scale = p.x_scale ? p.x_scale + full : nullptr;
            q.y_i32 = p.y_i32 ? p.y_i32 + full * p.N : nullptr;
            q.y_f32 = p.y_f32 ? p.y_f32 + full * p.N : nullptr;
            q.M = r;
            if (r <= 2) by2[n2++] = q;
            else if (r <= 4) by4[n4++] = q;
            else by8[n8++] = q;
        }
    }
    cudaError_t e = cudaSuccess;
    if (n8) e = launch_products<8>(by8, n8, err, s);
    if (e == cudaSuccess && n4) e = launch_products<4>(by4, n4, err, s);
    if (e == cudaSuccess && n2) e = launch_products<2>(by2, n2, err, s);
    return e;
}

}  // namespace trit

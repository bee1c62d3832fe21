// BITCOS weights: y = W x for one activation row with W stored as a presence
// bitmap and compacted signs ("BITCOS: Intel's Ternary LLM Weight Format Goes
// Below 1.58 Bits" -- A bitmap and a sign; Decoding is the other half of the
// bill), for comparison with the 2-bit planes.
//
// Layout (the blocked form: every row starts on a word of both arrays):
//   bitmap   uint64 [N][B], B = ceil(K/64): bit c%64 of word [r][c/64] is set
//            when W[r][c] != 0; bits past K are 0;
//   sign_off uint32 [N+1]: sign_off[0] = 0, sign_off[r+1] = sign_off[r] +
//            ceil(nnz_r / 32);
//   signs    uint32 [sign_off[N] + 2]: the k-th non-zero of row r (column
//            order) is -1 when bit k%32 of word sign_off[r] + k/32 is set.
//
// Decoding a 64-column word needs the signs of its set bits placed at those
// bits: a bit deposit, which sm_103a lacks.  The kernel deposits a byte at a
// time from a 64 KB table in shared memory, indexed by a presence byte and the
// next eight sign bits (the page's GPU decoder uses a table of presence and
// sign nibbles the same way), then runs the result through the same
// code-word multiply-accumulate as the bit-plane kernel: y = sum c x - sum x
// with c = 1 + pos - neg.
//
// One thread per row: it walks the row's bitmap words in order and reads its
// sign bits through a 64-bit cursor refilled 32 bits at a time, 32 columns per
// step so that one refill always suffices; both streams are loaded four words
// ahead, so no load waits on the decoding; the 32 rows of a warp move through the same columns
// together, so the staged activation words are read as broadcasts.  Persistent
// CTAs take contiguous ranges of the list's rows split by cost (bitmap words)
// and stage each product's activation row once.
#include <mutex>

#include "trit_internal.cuh"

namespace trit {
namespace {

constexpr int kWarpsB = 8;
constexpr int kThreadsB = kWarpsB * 32;
constexpr int kLutBytes = 65536;
constexpr int kMaxListB = TRIT_MAX_LIST_PER_LAUNCH;

struct BEntry {
    const uint64_t *bitmap;
    const uint32_t *sign_off;
    const uint32_t *signs;
    const int8_t *x;
    const float *x_scale;
    int32_t *y_i32;
    float *y_f32;
    int64_t N;
    int64_t sign_words;   // length of signs: every copy is clamped to it
    int64_t cost_begin;   // prefix sum of N * B over the list
    int32_t K, B;
    float w_scale;
    int32_t pad_;
};

struct BList {
    int32_t count;
    int32_t max_beats;    // staged activation beats
    int64_t total_cost;
    BEntry e[kMaxListB];
};
static_assert(sizeof(BList) <= 32764, "kernel parameter space");

// Deposit table: entry (m << 8) | s holds the low bits of s placed, in order,
// at the set bits of the byte m (the rest 0).  Uploaded once per device.
__device__ __align__(16) uint8_t g_deposit[kLutBytes];

// Code-word multiply-accumulate of one 32-column word pair against the
// permuted activation words (byte i of x[j] = column 8i + j): acc[j] gathers
// the 4^j-weighted codes of even word j, acc[4+j] of the odd ones.
__device__ __forceinline__ void mac_codes_b(uint32_t P, uint32_t N, const uint32_t *x, int (&acc)[8]) {
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

__device__ __forceinline__ int32_t codes_sum(const int (&acc)[8]) {
    return (acc[0] + acc[4]) + ((acc[1] + acc[5]) >> 2) + ((acc[2] + acc[6]) >> 4) +
           ((acc[3] + acc[7]) >> 6);
}

// Deposit the low bits of s into the set bits of the 32-bit word b, a byte at a time.
__device__ __forceinline__ uint32_t deposit32(uint32_t s, uint32_t b, const uint8_t *lut) {
    uint32_t n = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t mb = (b >> (8 * j)) & 0xFFu;
        n |= uint32_t(lut[(mb << 8) | (s & 0xFFu)]) << (8 * j);
        s >>= __popc(mb);
    }
    return n;
}

// Stage entry E's activation row (permuted, zero past K) and its column sum.
__device__ __forceinline__ int32_t stage_row(const BEntry &E, uint32_t *xs, int32_t *s_part) {
    const int halves = 2 * E.B;
    int32_t sum = 0;
    for (int hb = threadIdx.x; hb < halves; hb += kThreadsB) {
        const int c0 = hb * 32;
        const uint4 *p = reinterpret_cast<const uint4 *>(E.x + c0);
        const uint4 u0 = p[0], u1 = p[1];
        uint32_t in[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        if (c0 + 32 > E.K) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int lim = E.K - (c0 + 4 * q);
                const uint32_t keep = lim >= 4 ? 0xFFFFFFFFu : (lim <= 0 ? 0u : ((1u << (8 * lim)) - 1u));
                in[q] &= keep;
            }
        }
        uint32_t out[8];
        permute_block(in, out);
#pragma unroll
        for (int k = 0; k < 8; ++k) sum = dp4a_ss(in[k], 0x01010101u, sum);
        uint32_t *dst = xs + (hb >> 1) * kXBeatWords + (hb & 1) * 8;
        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(out[0], out[1], out[2], out[3]);
        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(~0u, sum, o);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = sum;
    __syncthreads();
    int32_t t = 0;
#pragma unroll
    for (int i = 0; i < kWarpsB; ++i) t += s_part[i];
    return t;
}

// First row of entry e whose cost is >= c (E.N when none is).
__device__ __forceinline__ int64_t first_row(const BEntry &E, int64_t c) {
    if (c <= E.cost_begin) return 0;
    const int64_t r = (c - E.cost_begin + E.B - 1) / E.B;
    return r < E.N ? r : E.N;
}

__global__ void __launch_bounds__(kThreadsB) bitcos_gemv_kernel(const __grid_constant__ BList L) {
    extern __shared__ __align__(16) uint8_t smem[];
    uint8_t *lut = smem;
    uint32_t *xs = reinterpret_cast<uint32_t *>(smem + kLutBytes);
    int32_t *s_part = reinterpret_cast<int32_t *>(xs + L.max_beats * kXBeatWords);

    for (int i = threadIdx.x; i < kLutBytes / 16; i += kThreadsB)
        reinterpret_cast<uint4 *>(lut)[i] = reinterpret_cast<const uint4 *>(g_deposit)[i];

    const int64_t begin = L.total_cost * blockIdx.x / gridDim.x;
    const int64_t end = L.total_cost * (blockIdx.x + 1) / gridDim.x;
    for (int e = 0; e < L.count; ++e) {
        const BEntry &E = L.e[e];
        const int64_t rb = first_row(E, begin), re = first_row(E, end);
        if (rb >= re) continue;
        __syncthreads();   // the previous entry's rows are done with xs (and lut is filled)
        const int32_t xsum = stage_row(E, xs, s_part);
        __syncthreads();
        const float xsc = *E.x_scale;
        const int B = E.B;
        for (int64_t row = rb + threadIdx.x; row < re; row += kThreadsB) {
            // the row's sign words, clamped to the array: nothing outside it is read
            const int64_t sw = E.sign_words;
            const int64_t o1 = E.sign_off[row + 1] < sw ? int64_t(E.sign_off[row + 1]) : sw;
            const int64_t o0 = E.sign_off[row] < o1 ? int64_t(E.sign_off[row]) : o1;
            const int64_t nw = o1 - o0;
            const uint32_t *sp = E.signs + o0;
            const uint64_t *bm = E.bitmap + row * B;
            uint64_t cur = 0;    // sign bits not yet used, lowest first
            int avail = 0;       // how many
            int acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            // both streams are read in order, so their next words are loaded four
            // ahead: bitmap words i..i+3 in b0..b3, the next sign words in q0..q3
            uint64_t b0 = __ldg(bm), b1 = B > 1 ? __ldg(bm + 1) : 0ull;
            uint64_t b2 = B > 2 ? __ldg(bm + 2) : 0ull, b3 = B > 3 ? __ldg(bm + 3) : 0ull;
            uint32_t q0 = nw > 0 ? __ldg(sp) : 0u, q1 = nw > 1 ? __ldg(sp + 1) : 0u;
            uint32_t q2 = nw > 2 ? __ldg(sp + 2) : 0u, q3 = nw > 3 ? __ldg(sp + 3) : 0u;
            int64_t nq = 4;      // the next sign word to load
            for (int i = 0; i < B; ++i) {
                const uint64_t b = b0;
                b0 = b1;
                b1 = b2;
                b2 = b3;
                b3 = i + 4 < B ? __ldg(bm + i + 4) : 0ull;
                const uint32_t *xw = xs + i * kXBeatWords;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint32_t bh = uint32_t(b >> (32 * h));
                    const int k = __popc(bh);
                    if (avail < k) {   // avail <= 31 here, so 32 more bits fit
                        cur |= uint64_t(q0) << avail;
                        avail += 32;
                        q0 = q1;
                        q1 = q2;
                        q2 = q3;
                        q3 = nq < nw ? __ldg(sp + nq) : 0u;
                        ++nq;
                    }
                    const uint32_t n = deposit32(uint32_t(cur), bh, lut);
                    cur >>= k;
                    avail -= k;
                    mac_codes_b(bh & ~n, n, xw + 8 * h, acc);
                }
            }
            const int32_t y = codes_sum(acc) - xsum;
            if (E.y_i32) E.y_i32[row] = y;
            if (E.y_f32) E.y_f32[row] = dequant(y, E.w_scale, xsc);
        }
    }
}

std::mutex g_table_mutex;
bool g_table_ready[64];

// Upload the deposit table to the current device once (synchronous).
cudaError_t ensure_table(int dev) {
    std::lock_guard<std::mutex> lock(g_table_mutex);
    if (g_table_ready[dev]) return cudaSuccess;
    static uint8_t host[kLutBytes];
    for (int i = 0; i < kLutBytes; ++i) {
        const uint32_t m = uint32_t(i) >> 8, sb = uint32_t(i) & 0xFFu;
        uint32_t r = 0, k = 0;
        for (int j = 0; j < 8; ++j)
            if ((m >> j) & 1u) {
                r |= ((sb >> k) & 1u) << j;
                ++k;
            }
        host[i] = uint8_t(r);
    }
    const cudaError_t e = cudaMemcpyToSymbol(g_deposit, host, sizeof host);
    if (e == cudaSuccess) g_table_ready[dev] = true;
    return e;
}

}  // namespace

int bitcos_pack_host(const int8_t *w, int64_t N, int64_t K, uint64_t *bitmap, uint32_t *sign_off,
                     uint32_t *signs, int64_t *sign_words) {
    const int64_t B = (K + 63) / 64;
    // pass 1: value check and the sign words
    int64_t words = 0;
    for (int64_t r = 0; r < N; ++r) {
        int64_t nnz = 0;
        const int8_t *row = w + r * K;
        for (int64_t c = 0; c < K; ++c) {
            if (row[c] < -1 || row[c] > 1) return TRIT_E_VALUE;
            nnz += row[c] != 0;
        }
        words += (nnz + 31) / 32;
    }
    if (words > int64_t(0xFFFFFFFFu) - 2) return TRIT_E_SHAPE;
    *sign_words = words + 2;
    if (!signs) return TRIT_OK;
    // pass 2: the arrays
    int64_t off = 0;
    sign_off[0] = 0;
    for (int64_t r = 0; r < N; ++r) {
        const int8_t *row = w + r * K;
        uint64_t *bm = bitmap + r * B;
        for (int64_t i = 0; i < B; ++i) bm[i] = 0;
        uint32_t acc = 0;
        int64_t k = 0;
        for (int64_t c = 0; c < K; ++c) {
            if (row[c] == 0) continue;
            bm[c >> 6] |= uint64_t(1) << (c & 63);
            if (row[c] < 0) acc |= 1u << (k & 31);
            if ((++k & 31) == 0) {
                signs[off++] = acc;
                acc = 0;
            }
        }
        if (k & 31) signs[off++] = acc;
        sign_off[r + 1] = uint32_t(off);
    }
    signs[off] = 0;
    signs[off + 1] = 0;
    return TRIT_OK;
}

cudaError_t launch_bitcos_many(const BitcosDev *list, int count, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    e = ensure_table(dev);
    if (e != cudaSuccess) return e;
    static thread_local BList L;
    int base = 0;
    while (base < count) {
        const int n = count - base < kMaxListB ? count - base : kMaxListB;
        L.count = n;
        int64_t cost = 0;
        int maxB = 1;
        for (int i = 0; i < n; ++i) {
            const BitcosDev &p = list[base + i];
            BEntry &E = L.e[i];
            E.bitmap = p.bitmap;
            E.sign_off = p.sign_off;
            E.signs = p.signs;
            E.x = p.x;
            E.x_scale = p.x_scale;
            E.y_i32 = p.y_i32;
            E.y_f32 = p.y_f32;
            E.N = p.N;
            E.sign_words = p.sign_words;
            E.K = int32_t(p.K);
            E.B = int32_t((p.K + 63) / 64);
            E.w_scale = p.w_scale;
            E.pad_ = 0;
            E.cost_begin = cost;
            cost += p.N * E.B;
            maxB = E.B > maxB ? E.B : maxB;
        }
        L.total_cost = cost;
        L.max_beats = maxB;
        const size_t smem = size_t(kLutBytes) + size_t(maxB) * kXBeatWords * 4 + kWarpsB * 4;
        e = cudaFuncSetAttribute(bitcos_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(smem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bitcos_gemv_kernel, kThreadsB, smem);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorInvalidConfiguration;
        if (cost > 0) {
            int64_t ctas = int64_t(per_sm) * device_sm_count();
            int64_t rows = 0;
            for (int i = 0; i < n; ++i) rows += L.e[i].N;
            ctas = ctas < rows ? ctas : rows;
            bitcos_gemv_kernel<<<unsigned(ctas), kThreadsB, smem, s>>>(L);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
        base += n;
    }
    return cudaSuccess;
}

}  // namespace trit

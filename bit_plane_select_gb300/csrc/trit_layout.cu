// Layout kernels: pack int8 ternary weights into .trit v1 bit planes, unpack
// them, and verify the two payload invariants.
//
// "The .trit format, version 1" -- 2.3 Ternary payload: beat b of row r is 16
// bytes at (r*B + b)*16, a little-endian u64 `pos` then `neg`, bit k <=> column
// 64b + k; P1 (pos & neg == 0) and P2 (padding bits past the last column clear,
// tail mask computed in 64 bits).
//
// One warp owns one beat in pack/unpack: lane i handles columns 64b+i and
// 64b+32+i, so a warp reads 2 x 32 consecutive int8 and the ballot of the
// lanes' predicates is the 32-bit plane word itself.
#include "trit_internal.cuh"

namespace trit {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__global__ void __launch_bounds__(kThreads) pack_kernel(const int8_t *__restrict__ w, int64_t N,
                                                        int64_t K, int64_t B,
                                                        uint4 *__restrict__ planes,
                                                        uint32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t total = N * B;
    bool bad = false;
    for (int64_t beat = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5); beat < total;
         beat += int64_t(gridDim.x) * kWarps) {
        const int64_t r = beat / B, b = beat - r * B;
        const int64_t c0 = b * 64 + lane, c1 = c0 + 32;
        const int8_t *row = w + r * K;
        const int v0 = c0 < K ? row[c0] : 0;
        const int v1 = c1 < K ? row[c1] : 0;
        const uint32_t p0 = __ballot_sync(~0u, v0 == 1), p1 = __ballot_sync(~0u, v1 == 1);
        const uint32_t n0 = __ballot_sync(~0u, v0 == -1), n1 = __ballot_sync(~0u, v1 == -1);
        bad |= (v0 < -1 || v0 > 1 || v1 < -1 || v1 > 1);
        if (lane == 0) planes[beat] = make_uint4(p0, p1, n0, n1);
    }
    if (__any_sync(~0u, bad) && lane == 0) atomicOr(err, TRIT_ERR_NOT_TERNARY);
}

__global__ void store_scale_kernel(float *dst, float v) { *dst = v; }

__global__ void __launch_bounds__(kThreads) unpack_kernel(const uint4 *__restrict__ planes,
                                                          int64_t N, int64_t K, int64_t B,
                                                          int8_t *__restrict__ w,
                                                          uint32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t total = N * B;
    bool bad = false;
    for (int64_t beat = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5); beat < total;
         beat += int64_t(gridDim.x) * kWarps) {
        const int64_t r = beat / B, b = beat - r * B;
        const uint4 v = planes[beat];
        bad |= ((v.x & v.z) | (v.y & v.w)) != 0;
        const int64_t c0 = b * 64 + lane, c1 = c0 + 32;
        const uint32_t bit = 1u << lane;
        // a both-set position decodes to 0
        const int8_t w0 = (v.x & bit) ? ((v.z & bit) ? 0 : 1) : ((v.z & bit) ? -1 : 0);
        const int8_t w1 = (v.y & bit) ? ((v.w & bit) ? 0 : 1) : ((v.w & bit) ? -1 : 0);
        if (c0 < K) w[r * K + c0] = w0;
        if (c1 < K) w[r * K + c1] = w1;
    }
    if (__any_sync(~0u, bad) && lane == 0) atomicOr(err, TRIT_ERR_P1);
}

// One thread per beat.  A violating bit's position is (r*B + b)*64 + k; the
// smallest over the launch goes to *first_bad through atomicMin.
__global__ void __launch_bounds__(kThreads) verify_kernel(const uint4 *__restrict__ planes,
                                                          int64_t N, int64_t K, int64_t B,
                                                          uint32_t *err,
                                                          unsigned long long *first_bad) {
    const int64_t total = N * B;
    const int rem = int(K % 64);
    const unsigned long long tail = rem == 0 ? ~0ull : ((1ull << rem) - 1ull);
    uint32_t kinds = 0;
    unsigned long long first = ~0ull;
    for (int64_t beat = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; beat < total;
         beat += int64_t(gridDim.x) * blockDim.x) {
        const uint4 v = planes[beat];
        const unsigned long long pos = (unsigned long long)v.x | ((unsigned long long)v.y << 32);
        const unsigned long long neg = (unsigned long long)v.z | ((unsigned long long)v.w << 32);
        unsigned long long badbits = pos & neg;
        if (badbits) kinds |= TRIT_ERR_P1;
        const int64_t b = beat % B;
        if (b == B - 1) {
            const unsigned long long dirty = (pos | neg) & ~tail;
            if (dirty) kinds |= TRIT_ERR_P2;
            badbits |= dirty;
        }
        if (badbits && first == ~0ull)
            first = (unsigned long long)beat * 64ull + (unsigned long long)(__ffsll((long long)badbits) - 1);
    }
    if (kinds) atomicOr(err, kinds);
    if (first_bad && first != ~0ull) atomicMin(first_bad, first);
}

int grid_for(int64_t items, int per_block) {
    const int64_t want = (items + per_block - 1) / per_block;
    const int64_t cap = int64_t(device_sm_count()) * 16;
    return int(want < 1 ? 1 : (want > cap ? cap : want));
}

}  // namespace

cudaError_t launch_pack(const int8_t *w, int64_t N, int64_t K, float w_scale, uint8_t *planes,
                        float *scale_out, uint32_t *err, cudaStream_t s) {
    const int64_t B = beats_per_row(K);
    pack_kernel<<<grid_for(N * B, kWarps), kThreads, 0, s>>>(w, N, K, B,
                                                            reinterpret_cast<uint4 *>(planes), err);
    if (scale_out) store_scale_kernel<<<1, 1, 0, s>>>(scale_out, w_scale);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t *planes, int64_t N, int64_t K, int8_t *w, uint32_t *err,
                          cudaStream_t s) {
    const int64_t B = beats_per_row(K);
    unpack_kernel<<<grid_for(N * B, kWarps), kThreads, 0, s>>>(
        reinterpret_cast<const uint4 *>(planes), N, K, B, w, err);
    return cudaGetLastError();
}

cudaError_t launch_verify(const uint8_t *planes, int64_t N, int64_t K, uint32_t *err,
                          unsigned long long *first_bad, cudaStream_t s) {
    const int64_t B = beats_per_row(K);
    verify_kernel<<<grid_for(N * B, kThreads), kThreads, 0, s>>>(
        reinterpret_cast<const uint4 *>(planes), N, K, B, err, first_bad);
    return cudaGetLastError();
}

}  // namespace trit

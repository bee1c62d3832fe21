// Per-token absmax int8 activation quantiser ("Tritium: One Weight Format for
// Ternary Inference ..." -- Numerics: per-token absmax codes, invariant under
// a uniform positive scale).  The pages print no formula; the reading:
//   a = max_c |x_c|, inv = 127/a (IEEE division), q = clamp(rint(x*inv), -127, 127),
//   x_scale = a; a = 0 -> q = 0, scale 0; a < 2^-96 -> x and a first scaled by 2^96
//   (exact) so 127/a stays finite; a NaN/Inf in the row -> TRIT_ERR_NONFINITE,
//   q = 0, scale 0.
// Output rows have stride K_pad = 64*ceil(K/64) with a zero tail ("The .trit
// format, version 1" -- 2.3: activation buffers sized beats_per_row*64).
//
// One CTA per activation row; a list of quantisations is one launch.
#include "trit_internal.cuh"

namespace trit {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxList = TRIT_MAX_LIST_PER_LAUNCH;

struct QuantList {
    int32_t count;
    int32_t pad_;
    uint32_t *err;
    int64_t row_begin[kMaxList + 1];   // prefix sum of M over the list
    trit_act act[kMaxList];
};

__global__ void __launch_bounds__(kThreads) quant_kernel(const __grid_constant__ QuantList L) {
    __shared__ uint32_t s_max[kThreads / 32];
    __shared__ uint32_t s_bad[kThreads / 32];
    const int64_t row_id = blockIdx.x;
    int e = 0;
    while (e + 1 < L.count && L.row_begin[e + 1] <= row_id) ++e;
    const trit_act &A = L.act[e];
    const int64_t m = row_id - L.row_begin[e];
    const int64_t K = A.K;
    const int64_t Kp = beats_per_row(K) * 64;
    const float *x = A.x + m * K;
    int8_t *q = A.x_i8 + m * Kp;

    // absmax as the largest bit pattern of |x| (non-negative floats order as integers)
    uint32_t amax = 0, bad = 0;
    for (int64_t c = threadIdx.x; c < K; c += kThreads) {
        const float v = x[c];
        bad |= !isfinite(v);
        const uint32_t bits = __float_as_uint(v) & 0x7fffffffu;
        amax = bits > amax ? bits : amax;
    }
    for (int o = 16; o; o >>= 1) {
        amax = max(amax, __shfl_xor_sync(~0u, amax, o));
        bad |= __shfl_xor_sync(~0u, bad, o);
    }
    if ((threadIdx.x & 31) == 0) {
        s_max[threadIdx.x >> 5] = amax;
        s_bad[threadIdx.x >> 5] = bad;
    }
    __syncthreads();
    amax = 0;
    bad = 0;
#pragma unroll
    for (int i = 0; i < kThreads / 32; ++i) {
        amax = max(amax, s_max[i]);
        bad |= s_bad[i];
    }
    const float a = __uint_as_float(amax);

    if (bad || amax == 0) {
        for (int64_t c = threadIdx.x; c < Kp; c += kThreads) q[c] = 0;
        if (threadIdx.x == 0) {
            A.x_scale[m] = 0.0f;
            if (bad) atomicOr(L.err, TRIT_ERR_NONFINITE);
        }
        return;
    }
    const float pre = a < 0x1p-96f ? 0x1p96f : 1.0f;
    const float inv = __fdiv_rn(127.0f, __fmul_rn(a, pre));
    for (int64_t c = threadIdx.x; c < Kp; c += kThreads) {
        int v = 0;
        if (c < K) {
            v = __float2int_rn(__fmul_rn(__fmul_rn(x[c], pre), inv));
            v = v > 127 ? 127 : (v < -127 ? -127 : v);
        }
        q[c] = (int8_t)v;
    }
    if (threadIdx.x == 0) A.x_scale[m] = a;
}

}  // namespace

cudaError_t launch_quant_many(const trit_act *list, int count, uint32_t *err, cudaStream_t s) {
    for (int base = 0; base < count; base += kMaxList) {
        const int n = count - base < kMaxList ? count - base : kMaxList;
        QuantList L;
        L.count = n;
        L.pad_ = 0;
        L.err = err;
        L.row_begin[0] = 0;
        for (int i = 0; i < n; ++i) {
            L.act[i] = list[base + i];
            L.row_begin[i + 1] = L.row_begin[i] + list[base + i].M;
        }
        const int64_t rows = L.row_begin[n];
        // grid.x holds up to 2^31-1 blocks; longer lists were rejected on the host
        quant_kernel<<<dim3((unsigned)rows), kThreads, 0, s>>>(L);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace trit

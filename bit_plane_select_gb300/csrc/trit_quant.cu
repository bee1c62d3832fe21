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
// One CTA per activation row; the row is held in registers between the absmax
// reduction and the code pass (V float4 per thread), so it is read from memory
// once.  Rows longer than the register budget take a two-pass loop.  A list of
// quantisations is one launch.
#include "trit_internal.cuh"

namespace trit {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxList = TRIT_MAX_LIST_PER_LAUNCH;
constexpr int kMaxV = 8;     // float4 per thread held in registers: K_pad <= 8192

struct QuantList {
    int32_t count;
    int32_t pad_;
    uint32_t *err;
    int64_t row_begin[kMaxList + 1];   // prefix sum of M over the list
    trit_act act[kMaxList];
};

__device__ __forceinline__ int find_entry(const QuantList &L, int64_t row) {
    int lo = 0, hi = L.count - 1;   // largest e with row_begin[e] <= row
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (L.row_begin[mid] <= row) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Block-wide max of the |x| bit patterns and OR of the non-finite flags.
__device__ __forceinline__ void block_reduce(uint32_t &amax, uint32_t &bad) {
    __shared__ uint32_t s_max[kThreads / 32], s_bad[kThreads / 32];
#pragma unroll
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
}

// V > 0: the row lives in registers (V float4 per thread); V == 0: two passes.
template <int V>
__global__ void __launch_bounds__(kThreads) quant_kernel(const __grid_constant__ QuantList L) {
    const int64_t row_id = blockIdx.x;
    const trit_act &A = L.act[find_entry(L, row_id)];
    const int64_t m = row_id - L.row_begin[find_entry(L, row_id)];
    const int64_t K = A.K;
    const int64_t Kp = beats_per_row(K) * 64;
    const float *x = A.x + m * K;
    uint32_t *q4 = reinterpret_cast<uint32_t *>(A.x_i8 + m * Kp);   // K_pad % 64 == 0
    const bool vec = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(A.x) & 15) == 0);

    uint32_t amax = 0, bad = 0;
    float4 r[V > 0 ? V : 1];
    if constexpr (V > 0) {
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int64_t c = (int64_t(threadIdx.x) + i * kThreads) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (vec) {
                if (c < K) v = *reinterpret_cast<const float4 *>(x + c);
            } else {
                if (c + 0 < K) v.x = x[c + 0];
                if (c + 1 < K) v.y = x[c + 1];
                if (c + 2 < K) v.z = x[c + 2];
                if (c + 3 < K) v.w = x[c + 3];
            }
            r[i] = v;
        }
#pragma unroll
        for (int i = 0; i < V; ++i) {
            bad |= !isfinite(r[i].x) | !isfinite(r[i].y) | !isfinite(r[i].z) | !isfinite(r[i].w);
            amax = max(amax, max(max(quant_abs_bits(r[i].x), quant_abs_bits(r[i].y)),
                                 max(quant_abs_bits(r[i].z), quant_abs_bits(r[i].w))));
        }
    } else {
        for (int64_t c = threadIdx.x; c < K; c += kThreads) {
            const float v = x[c];
            bad |= !isfinite(v);
            amax = max(amax, quant_abs_bits(v));
        }
    }
    block_reduce(amax, bad);
    const QuantScale qs = quant_scale(amax, bad != 0);

    if constexpr (V > 0) {
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int64_t c = (int64_t(threadIdx.x) + i * kThreads) * 4;
            if (c < Kp) {
                // columns >= K hold 0 and code to 0
                q4[c / 4] = pack4(quant_code(r[i].x, qs), quant_code(r[i].y, qs),
                                  quant_code(r[i].z, qs), quant_code(r[i].w, qs));
            }
        }
    } else {
        for (int64_t c4 = threadIdx.x; c4 < Kp / 4; c4 += kThreads) {
            int v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t c = c4 * 4 + k;
                v[k] = c < K ? quant_code(x[c], qs) : 0;
            }
            q4[c4] = pack4(v[0], v[1], v[2], v[3]);
        }
    }
    if (threadIdx.x == 0) {
        A.x_scale[m] = qs.a;
        if (bad) atomicOr(L.err, TRIT_ERR_NONFINITE);
    }
}

template <int V>
cudaError_t launch_v(const QuantList &L, int64_t rows, cudaStream_t s) {
    quant_kernel<V><<<dim3((unsigned)rows), kThreads, 0, s>>>(L);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_many(const trit_act *list, int count, uint32_t *err, cudaStream_t s) {
    static thread_local QuantList L;
    for (int base = 0; base < count; base += kMaxList) {
        const int n = count - base < kMaxList ? count - base : kMaxList;
        L.count = n;
        L.pad_ = 0;
        L.err = err;
        L.row_begin[0] = 0;
        int64_t maxKp = 64;
        for (int i = 0; i < n; ++i) {
            L.act[i] = list[base + i];
            L.row_begin[i + 1] = L.row_begin[i] + list[base + i].M;
            const int64_t kp = beats_per_row(list[base + i].K) * 64;
            maxKp = kp > maxKp ? kp : maxKp;
        }
        const int64_t rows = L.row_begin[n];   // <= 2^31 - 1, checked on the host
        const int64_t per_thread = (maxKp + 4 * kThreads - 1) / (4 * kThreads);
        cudaError_t e;
        if (per_thread <= 1) e = launch_v<1>(L, rows, s);
        else if (per_thread <= 2) e = launch_v<2>(L, rows, s);
        else if (per_thread <= 4) e = launch_v<4>(L, rows, s);
        else if (per_thread <= kMaxV) e = launch_v<kMaxV>(L, rows, s);
        else e = launch_v<0>(L, rows, s);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace trit

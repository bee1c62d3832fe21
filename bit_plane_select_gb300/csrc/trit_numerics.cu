// Numerics epilogues around the ternary products ("Tritium: One Weight Format
// for Ternary Inference ..." -- Numerics):
//
//  - Folded: the normalisation's 1/rms never touches the elements.  Absmax
//    codes are unchanged by a uniform positive scale, so the codes are those of
//    u = x (.) g, computed with the quantiser's own arithmetic, and the rms
//    (sqrt(mean(x^2) + eps), in double) only divides the row's scale.
//  - IntMlp: relu(g)^2 u of the gate and up outputs equals t K with the integer
//    t = relu(a_g)^2 a_u and the uniform K = S_g^2 S_u, so the squared-ReLU
//    stage stays integer: t is formed exactly (128-bit), the next projection's
//    codes are round-half-even(127 t / max|t|) as an exact rational, and the
//    row's scale is max|t| K.
//
// One CTA per row, two passes over the row (the second re-reads from L1/L2).
//
// Also: the exhaustive device check of div127_rn, the division used by every
// fp32 dequantisation.
#include "trit_internal.cuh"

namespace trit {
namespace {

constexpr int kNThreads = 256;
constexpr int kNWarps = kNThreads / 32;
// IntMlp rows when there are no more rows than SMs (decode): one CTA per row
#ifndef TRIT_INTMLP_THREADS_FEW
#define TRIT_INTMLP_THREADS_FEW 1024
#endif
constexpr int kIntMlpThreadsFew = TRIT_INTMLP_THREADS_FEW;

__device__ __forceinline__ double block_sum_f64(double v, double *red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(~0u, v, o);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    double s = 0.0;
    for (int i = 0; i < kNWarps; ++i) s += red[i];   // same order in every thread
    return s;
}

// ---- Folded ----------------------------------------------------------------------

__global__ void __launch_bounds__(kNThreads) quant_folded_kernel(const float *x, const float *g,
                                                                 int64_t M, int64_t K, float eps,
                                                                 int64_t ldq, int8_t *q,
                                                                 float *x_scale, uint32_t *err) {
    __shared__ double red[kNWarps];
    __shared__ uint32_t redu[2][kNWarps];
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const float *xr = x + m * K;
        uint32_t amax = 0, bad = 0;
        double s2 = 0.0;
        for (int64_t c = threadIdx.x; c < K; c += kNThreads) {
            const float xv = xr[c];
            const float u = __fmul_rn(xv, g[c]);
            bad |= !isfinite(u);
            amax = max(amax, quant_abs_bits(u));
            s2 = __dadd_rn(s2, __dmul_rn(double(xv), double(xv)));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            amax = max(amax, __shfl_xor_sync(~0u, amax, o));
            bad |= __shfl_xor_sync(~0u, bad, o);
        }
        if ((threadIdx.x & 31) == 0) {
            redu[0][threadIdx.x >> 5] = amax;
            redu[1][threadIdx.x >> 5] = bad;
        }
        const double sum2 = block_sum_f64(s2, red);   // includes a barrier
        amax = 0;
        bad = 0;
        for (int i = 0; i < kNWarps; ++i) {
            amax = max(amax, redu[0][i]);
            bad |= redu[1][i];
        }
        const QuantScale qs = quant_scale(amax, bad != 0);
        int8_t *qr = q + m * ldq;
        for (int64_t c = threadIdx.x; c < ldq; c += kNThreads)
            qr[c] = c < K ? int8_t(quant_code(__fmul_rn(xr[c], g[c]), qs)) : int8_t(0);
        if (threadIdx.x == 0) {
            float s = 0.0f;
            if (!qs.zero) {
                const double rms = __dsqrt_rn(__dadd_rn(__ddiv_rn(sum2, double(K)), double(eps)));
                s = __double2float_rn(__ddiv_rn(double(qs.a), rms));
            }
            x_scale[m] = s;
            if (bad) atomicOr(err, TRIT_ERR_NONFINITE);
        }
        __syncthreads();   // red / redu reused by the next row
    }
}

// ---- IntMlp ----------------------------------------------------------------------

// NT threads per row (one CTA per row): a decode row (M = 1, N = 6,912) is
// latency-bound, so the row's first kHoldI * (NT - 32) columns are loaded once,
// held in registers through both passes, and the block maximum is reduced by
// one warp and broadcast.  The last warp takes no columns: it forms the
// scale, whose double arithmetic is slow on this device -- the factor
// S_g^2 S_u while the others reduce max|t|, the product with max|t| while they
// form the codes.
constexpr int kHoldI = 8;
template <int NT>
__global__ void __launch_bounds__(NT) intmlp_quant_kernel(const int32_t *ag, const int32_t *au,
                                                          int64_t M, int64_t N, int64_t ldq,
                                                          float w_g, float w_u,
                                                          const float *x_scale, int8_t *q,
                                                          float *h_scale) {
    constexpr int kW = NT / 32;
    constexpr int kC = NT - 32;   // threads that take columns
    static_assert(kW <= 32 && kW >= 2, "one warp reduces the warps' maxima");
    __shared__ uint64_t red[2][kW];
    __shared__ uint64_t fin[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // launched with programmatic serialisation: the next launch may start its
    // own set-up now; the gate and up outputs are read after the preceding grid
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    auto umax = [](uint64_t &hi, uint64_t &lo, uint64_t h2, uint64_t l2) {
        if (h2 > hi || (h2 == hi && l2 > lo)) {
            hi = h2;
            lo = l2;
        }
    };
    auto warp_max = [&](uint64_t &hi, uint64_t &lo) {
#pragma unroll
        for (int o = 16; o; o >>= 1)
            umax(hi, lo, __shfl_xor_sync(~0u, hi, o), __shfl_xor_sync(~0u, lo, o));
    };
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const int32_t *gr = ag + m * N, *ur = au + m * N;
        const bool scaler = warp == kW - 1;
        // the scaler warp's columns lie past every row (t = 0, code 0)
        const int64_t c0 = scaler ? INT64_MAX / 2 : int64_t(threadIdx.x);
        double kfac = 0.0;
        if (scaler && lane == 0) kfac = intmlp_scale_factor(w_g, w_u, x_scale[m]);
        int32_t g[kHoldI], u[kHoldI];
#pragma unroll
        for (int r = 0; r < kHoldI; ++r) {
            const int64_t c = int64_t(r) * kC + c0;
            g[r] = c < N ? gr[c] : 0;   // past N: t = 0, code 0
            u[r] = c < N ? ur[c] : 0;
        }
        trit_u128 amax = 0;
#pragma unroll
        for (int r = 0; r < kHoldI; ++r) {
            bool neg;
            const trit_u128 t = intmlp_abs_t(g[r], u[r], neg);
            amax = t > amax ? t : amax;
        }
        for (int64_t c = int64_t(kHoldI) * kC + c0; c < N; c += kC) {
            bool neg;
            const trit_u128 t = intmlp_abs_t(gr[c], ur[c], neg);
            amax = t > amax ? t : amax;
        }
        uint64_t hi = uint64_t(amax >> 64), lo = uint64_t(amax);
        warp_max(hi, lo);
        if (lane == 0) {
            red[0][warp] = hi;
            red[1][warp] = lo;
        }
        __syncthreads();
        if (warp == 0) {
            hi = lane < kW ? red[0][lane] : 0;
            lo = lane < kW ? red[1][lane] : 0;
            warp_max(hi, lo);
            if (lane == 0) {
                fin[0] = hi;
                fin[1] = lo;
            }
        }
        __syncthreads();
        hi = fin[0];
        lo = fin[1];
        if (scaler) {
            if (lane == 0) h_scale[m] = intmlp_scale_apply(hi, lo, kfac);
        } else {
            const IntMlpRow R = intmlp_row(hi, lo);
            int8_t *qr = q + m * ldq;
#pragma unroll
            for (int r = 0; r < kHoldI; r += 4) {
                const uint32_t w = intmlp_codes4(make_int4(g[r], g[r + 1], g[r + 2], g[r + 3]),
                                                 make_int4(u[r], u[r + 1], u[r + 2], u[r + 3]), R);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t c = int64_t(r + j) * kC + c0;
                    if (c < ldq) qr[c] = int8_t(w >> (8 * j));
                }
            }
            for (int64_t c = int64_t(kHoldI) * kC + c0; c < ldq; c += kC)
                qr[c] = c < N ? int8_t(intmlp_code_est(gr[c], ur[c], R)) : int8_t(0);
        }
        __syncthreads();   // red and fin reused by the next row
    }
}

// ---- division by 127 --------------------------------------------------------------

// Every float32 bit pattern i in [lo, hi): count those where div127_rn(f) and
// the IEEE divide disagree (NaN results agree with any NaN).
__global__ void __launch_bounds__(256) check_div127_kernel(uint64_t lo, uint64_t hi,
                                                           unsigned long long *mismatches) {
    unsigned long long bad = 0;
    const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
    for (uint64_t i = lo + uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < hi; i += stride) {
        const float f = __uint_as_float(uint32_t(i));
        const float a = div127_rn(f), b = __fdiv_rn(f, 127.0f);
        bad += (__float_as_uint(a) != __float_as_uint(b)) && !(isnan(a) && isnan(b));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) bad += __shfl_xor_sync(~0u, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(mismatches, bad);
}

int rows_grid(int64_t M) {
    const int64_t cap = int64_t(device_sm_count()) * 8;
    return int(M < cap ? M : cap);
}

// ---- max|t| partials ---------------------------------------------------------------

constexpr int kMaxTmaxJobs = 32;
struct TmaxJobs {
    MlpTmaxJob job[kMaxTmaxJobs];
    int64_t warp_begin[kMaxTmaxJobs + 1];   // prefix sums of ceil(F / 32)
    int32_t count;
};

// One warp per partial: lane l takes column 32k + l of its block and also
// stores its signed fp32 product (the workspace layout of mlp_tmax_bytes).  Launched
// with programmatic serialisation: the gate and up outputs are read after the
// preceding grid.
__global__ void __launch_bounds__(256) mlp_tmax_kernel(const __grid_constant__ TmaxJobs J) {
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t gw = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= J.warp_begin[J.count]) return;   // whole warps only: no block barrier follows
    int j = 0;
    while (j + 1 < J.count && J.warp_begin[j + 1] <= gw) ++j;
    const MlpTmaxJob &B = J.job[j];
    const int64_t k = gw - J.warp_begin[j];
    const int64_t c = 32 * k + lane;
    bool neg;
    const trit_u128 t = c < B.F ? intmlp_abs_t(B.a_gate[c], B.a_up[c], neg) : trit_u128(0);
    uint64_t hi = uint64_t(t >> 64), lo = uint64_t(t);
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const uint64_t h2 = __shfl_xor_sync(~0u, hi, o), l2 = __shfl_xor_sync(~0u, lo, o);
        if (h2 > hi || (h2 == hi && l2 > lo)) {
            hi = h2;
            lo = l2;
        }
    }
    if (lane == 0) {
        B.tmax[2 * k] = hi;
        B.tmax[2 * k + 1] = lo;
    }
    // the column's signed fp32 product, for the down launch's codes (0 past F)
    mlp_tf_of(B.tmax, (B.F + 31) / 32)[c] = c < B.F ? intmlp_tf(B.a_gate[c], B.a_up[c]) : 0.0f;
}

}  // namespace

cudaError_t launch_mlp_tmax(const MlpTmaxJob *jobs, int n, cudaStream_t s) {
    static thread_local TmaxJobs J;
    for (int base = 0; base < n; base += kMaxTmaxJobs) {
        const int m = n - base < kMaxTmaxJobs ? n - base : kMaxTmaxJobs;
        J.count = m;
        J.warp_begin[0] = 0;
        for (int i = 0; i < m; ++i) {
            J.job[i] = jobs[base + i];
            J.warp_begin[i + 1] = J.warp_begin[i] + (jobs[base + i].F + 31) / 32;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned((J.warp_begin[m] + 7) / 8));
        cfg.blockDim = dim3(256);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, mlp_tmax_kernel, J);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_quant_folded(const float *x, const float *g, int64_t M, int64_t K, float eps,
                                int8_t *q, float *x_scale, uint32_t *err, cudaStream_t s) {
    const int64_t ldq = beats_per_row(K) * 64;
    quant_folded_kernel<<<rows_grid(M), kNThreads, 0, s>>>(x, g, M, K, eps, ldq, q, x_scale, err);
    return cudaGetLastError();
}

cudaError_t launch_check_div127(uint64_t lo, uint64_t hi, unsigned long long *mismatches,
                                cudaStream_t s) {
    check_div127_kernel<<<device_sm_count() * 8, 256, 0, s>>>(lo, hi, mismatches);
    return cudaGetLastError();
}

cudaError_t launch_intmlp_quant(const int32_t *ag, const int32_t *au, int64_t M, int64_t N,
                                float w_g, float w_u, const float *x_scale, int8_t *q,
                                float *h_scale, cudaStream_t s) {
    const int64_t ldq = beats_per_row(N) * 64;
    const bool few = M <= int64_t(device_sm_count());
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(few ? int(M) : rows_grid(M)));
    cfg.blockDim = dim3(few ? kIntMlpThreadsFew : kNThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (few)
        return cudaLaunchKernelEx(&cfg, intmlp_quant_kernel<kIntMlpThreadsFew>, ag, au, M, N, ldq,
                                  w_g, w_u, x_scale, q, h_scale);
    return cudaLaunchKernelEx(&cfg, intmlp_quant_kernel<kNThreads>, ag, au, M, N, ldq, w_g, w_u,
                              x_scale, q, h_scale);
}

}  // namespace trit

// Read-bandwidth probe: streams a device buffer once with 16-byte loads that
// bypass L1 (the access the select-accumulate kernels use for the planes) and
// reduces what it read into one word, so the loads cannot be elided.  It is
// the same-run denominator the benchmark reports next to the measured copy
// rate: how fast this device reads HBM with a plain, fully coalesced stream.
#include "trit_internal.cuh"

namespace trit {
namespace {

__global__ void __launch_bounds__(256) read_probe_kernel(const uint4 *p, int64_t n16, uint32_t *sink) {
    uint32_t acc = 0;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {   // four loads in flight per thread
        const uint4 a = ldg_stream(p + i), b = ldg_stream(p + i + stride);
        const uint4 c = ldg_stream(p + i + 2 * stride), d = ldg_stream(p + i + 3 * stride);
        acc ^= a.x ^ a.y ^ a.z ^ a.w ^ b.x ^ b.y ^ b.z ^ b.w ^ c.x ^ c.y ^ c.z ^ c.w ^ d.x ^ d.y ^
               d.z ^ d.w;
    }
    for (; i < n16; i += stride) {
        const uint4 a = ldg_stream(p + i);
        acc ^= a.x ^ a.y ^ a.z ^ a.w;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) acc ^= __shfl_xor_sync(~0u, acc, o);
    if ((threadIdx.x & 31) == 0 && acc == 0x9E3779B9u) atomicXor(sink, acc);   // almost never taken
}

// ---- issue-rate probe ----------------------------------------------------------
// How many of one instruction an SM completes per clock: every thread runs
// eight independent chains of the instruction, 32 per loop trip, and thread 0
// of each CTA records (SM id, clock64 at the start, clock64 at the end) once
// all its warps have passed the matching barrier.  The shared-memory kinds
// read conflict-free addresses (lane-contiguous words / 16-byte vectors) and
// fold what they read into the chains, so no load is dead.
template <int KIND, int U>
__device__ __forceinline__ void probe_op(uint32_t (&a)[8], uint32_t b, uint32_t c, uint32_t smb,
                                         uint32_t zmask) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        if constexpr (KIND == TRIT_PROBE_DP4A) {
            asm volatile("dp4a.s32.s32 %0, %1, %2, %0;" : "+r"(a[k]) : "r"(b), "r"(c));
        } else if constexpr (KIND == TRIT_PROBE_LOP3) {
            asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(a[k]) : "r"(b), "r"(c));
        } else if constexpr (KIND == TRIT_PROBE_PRMT) {
            asm volatile("prmt.b32 %0, %0, %1, %2;" : "+r"(a[k]) : "r"(b), "r"(c));
        } else if constexpr (KIND == TRIT_PROBE_SHF) {
            asm volatile("shf.l.wrap.b32 %0, %0, %1, %2;" : "+r"(a[k]) : "r"(b), "r"(c));
        } else if constexpr (KIND == TRIT_PROBE_IMAD) {
            asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(a[k]) : "r"(b), "r"(c));
        } else if constexpr (KIND == TRIT_PROBE_IADD) {
            asm volatile("add.u32 %0, %0, %1;" : "+r"(a[k]) : "r"(b));
        } else if constexpr (KIND == TRIT_PROBE_SHFL) {
            asm volatile("shfl.sync.bfly.b32 %0, %0, 1, 0x1f, 0xffffffff;" : "+r"(a[k]));
        } else if constexpr (KIND == TRIT_PROBE_DP4A_SU) {
            asm volatile("dp4a.s32.u32 %0, %1, %2, %0;" : "+r"(a[k]) : "r"(b), "r"(c));
        } else if constexpr (KIND == TRIT_PROBE_DP4A_LOP3) {
            asm volatile("dp4a.s32.s32 %0, %1, %2, %0;" : "+r"(a[k]) : "r"(b), "r"(c));
            asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(a[k]) : "r"(b), "r"(c));
        } else {
            // each load's address carries a zero the compiler cannot see (the
            // chain value and-ed with a mask that is 0 at run time), so no load
            // can be hoisted out of the loop and a thread has at most eight in
            // flight
            const uint32_t z = a[k] & zmask;
            if constexpr (KIND == TRIT_PROBE_LDS32) {
                // smb = shared base + 4 * lane: word (lane, block 8U + k) of 32 x 32 words
                uint32_t v;
                asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(smb + z + 128u * (8 * U + k)));
                a[k] ^= v;
            } else {   // TRIT_PROBE_LDS128: smb = shared base + 16 * lane, blocks of 512 bytes
                asm volatile(
                    "{\n\t.reg .b32 t0, t1, t2, t3;\n\t"
                    "ld.volatile.shared.v4.u32 {t0, t1, t2, t3}, [%1];\n\t"
                    "xor.b32 t0, t0, t1;\n\txor.b32 t2, t2, t3;\n\t"
                    "xor.b32 t0, t0, t2;\n\txor.b32 %0, %0, t0;\n\t}"
                    : "+r"(a[k])
                    : "r"(smb + z + 512u * (8 * U + k)));
            }
        }
    }
}

template <int KIND>
__global__ void __launch_bounds__(512) issue_probe_kernel(int64_t iters, uint32_t seed, uint32_t zmask,
                                                           uint32_t *sink, unsigned long long *rec) {
    __shared__ __align__(16) uint32_t sm[4 * 32 * 32];   // 16 KB: 32 blocks of 32 lanes x 16 bytes
    for (int i = threadIdx.x; i < 4 * 32 * 32; i += blockDim.x) sm[i] = seed ^ (uint32_t(i) * 0x9E3779B9u);
    const int lane = threadIdx.x & 31;
    uint32_t a[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) a[k] = seed + threadIdx.x * 8u + k;
    const uint32_t b = seed * 3u + 1u, c = (seed ^ 0x5410u) & 0x771fu;
    const uint32_t smb = uint32_t(__cvta_generic_to_shared(sm)) +
                         uint32_t(lane) * (KIND == TRIT_PROBE_LDS128 ? 16u : 4u);
    __syncthreads();
    const unsigned long long t0 = clock64();
    for (int64_t it = 0; it < iters; ++it) {
        probe_op<KIND, 0>(a, b, c, smb, zmask);
        probe_op<KIND, 1>(a, b, c, smb, zmask);
        probe_op<KIND, 2>(a, b, c, smb, zmask);
        probe_op<KIND, 3>(a, b, c, smb, zmask);
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    uint32_t x = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) x ^= a[k];
    if (x == 0x9E3779B9u) atomicXor(sink, x);   // almost never taken; keeps the chains live
    if (threadIdx.x == 0) {
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        rec[3 * blockIdx.x + 0] = smid;
        rec[3 * blockIdx.x + 1] = t0;
        rec[3 * blockIdx.x + 2] = t1;
    }
}

}  // namespace

cudaError_t launch_issue_probe(int kind, int blocks, int threads, int64_t iters, uint32_t *sink,
                               unsigned long long *rec, cudaStream_t s) {
    const uint32_t seed = 0x2545F491u;
    switch (kind) {
#define TRIT_PROBE_CASE(K) \
    case K: issue_probe_kernel<K><<<blocks, threads, 0, s>>>(iters, seed, 0u, sink, rec); break;
        TRIT_PROBE_CASE(TRIT_PROBE_DP4A)
        TRIT_PROBE_CASE(TRIT_PROBE_LOP3)
        TRIT_PROBE_CASE(TRIT_PROBE_PRMT)
        TRIT_PROBE_CASE(TRIT_PROBE_SHF)
        TRIT_PROBE_CASE(TRIT_PROBE_IMAD)
        TRIT_PROBE_CASE(TRIT_PROBE_IADD)
        TRIT_PROBE_CASE(TRIT_PROBE_SHFL)
        TRIT_PROBE_CASE(TRIT_PROBE_LDS32)
        TRIT_PROBE_CASE(TRIT_PROBE_LDS128)
        TRIT_PROBE_CASE(TRIT_PROBE_DP4A_LOP3)
        TRIT_PROBE_CASE(TRIT_PROBE_DP4A_SU)
#undef TRIT_PROBE_CASE
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_read_probe(const void *p, int64_t bytes, uint32_t *sink, cudaStream_t s) {
    const int64_t n16 = bytes / 16;
    read_probe_kernel<<<device_sm_count() * 8, 256, 0, s>>>(reinterpret_cast<const uint4 *>(p), n16,
                                                            sink);
    return cudaGetLastError();
}

}  // namespace trit

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

}  // namespace

cudaError_t launch_read_probe(const void *p, int64_t bytes, uint32_t *sink, cudaStream_t s) {
    const int64_t n16 = bytes / 16;
    read_probe_kernel<<<device_sm_count() * 8, 256, 0, s>>>(reinterpret_cast<const uint4 *>(p), n16,
                                                            sink);
    return cudaGetLastError();
}

}  // namespace trit

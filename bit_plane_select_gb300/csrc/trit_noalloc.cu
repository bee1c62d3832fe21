// Fixed device scratch for trit_gemm_noalloc: a file-scope buffer that is part
// of the library's device image, so that calls through that entry point never
// allocate.  Its address differs per device (each context that loads the image
// gets its own copy) and is looked up once per device on first use.
#include <mutex>

#include "trit_internal.cuh"

static __device__ __align__(256) uint8_t trit_fixed_scratch[TRIT_NOALLOC_SCRATCH_BYTES];

namespace trit {

namespace {
constexpr int kScratchDevices = 64;
void *g_scratch_addr[kScratchDevices] = {nullptr};
std::mutex g_scratch_mutex;
}  // namespace

// Address of this device's copy of the buffer.  The first call on a device runs
// cudaGetSymbolAddress with that device current (which may load the image);
// later calls read the cached address.
cudaError_t fixed_scratch(uint8_t **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, trit_fixed_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = static_cast<uint8_t *>(g_scratch_addr[dev]);
    return cudaSuccess;
}

}  // namespace trit

// Shared-memory, mbarrier, tensor-core and copy wrappers used by the two
// tensor-core kernels (trit_prefill.cu: CTA pairs for many activation rows;
// trit_skinny.cu: single CTAs for a few), and the fp16 activation copy both
// contract against.
//
// Both kernels contract int8 activations with +-1 weights as fp16 operands of
// tcgen05.mma kind::f16 with fp32 accumulators, exact for K < 131072 (every
// partial sum is an integer of magnitude <= 127*K < 2^24).  Operands live in
// shared memory as 128-byte-swizzled K-major tiles of 64 columns (one plane
// beat): row r, 16-byte chunk c at (r/8)*1024 + (r%8)*128 + ((c ^ r%8) * 16).
// Inside a beat the columns are permuted identically on both sides (word k of
// half h holds columns 32h+k and 32h+k+16), which leaves the contraction
// unchanged.
#pragma once

#include "trit_internal.cuh"

namespace trit {
namespace tc {

constexpr int kBK = 64;                                   // columns per stage (one beat)
constexpr unsigned long long kWaitNs = 4000000000ull;     // bound of every mbarrier wait: 4 s

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.shared::cta.b64 st, [%0];\n}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of the given parity (acquire at cluster scope: some arrivals
// come from the peer CTA); false after kWaitNs (then *timed_out is set).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint32_t *timed_out) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (*reinterpret_cast<volatile uint32_t *>(timed_out)) return false;
        if (global_ns() - t0 > kWaitNs) {
            atomicExch(timed_out, 1u);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}


// 128-byte-swizzled K-major shared-memory matrix descriptor (version 1): start
// address, leading offset 16 B (unused for this layout), stride 1024 B between
// groups of eight 128-byte rows.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t(1) << 16) | (uint64_t(1024 >> 4) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// 16-byte asynchronous global -> shared copy through L2; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{\n .reg .b64 st;\n mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
// 1-D bulk copy global -> shared completing on an mbarrier (16-byte aligned,
// size a multiple of 16).
__device__ __forceinline__ void bulk_load(void *sdst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major tile.
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
    return uint32_t((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}


// 8 fp16x2 words (cols 32h + k and 32h + k + 16, k = k0..k0+7, k0 = 0 or 8) of one
// plane half; for k0 = 8 the caller passes the words shifted right by 8.
__device__ __forceinline__ void expand_quarter(uint32_t P, uint32_t N, uint32_t (&w)[8]) {
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const uint32_t m = 0x00010001u << s;
        w[s] = (P & m) * (0x3C00u >> s) + (N & m) * (0xBC00u >> s);
    }
}

// 16 fp16x2 words of activation columns 32h..32h+31 (natural int8 words in[0..7]).
__device__ __forceinline__ void convert_half(const uint32_t (&in)[8], uint32_t (&w)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t u = in[q] ^ 0x80808080u, v = in[q + 4] ^ 0x80808080u;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t t = prmt(u, v, uint32_t(i) | (uint32_t(4 + i) << 8));
            const uint32_t h = (t & 0x00FF00FFu) | 0x64006400u;   // 1024 + (x + 128)
            w[4 * q + i] = hsub2(h, 0x64806480u);                // minus 1152
        }
    }
}

// ---- the fp16 activation copy ---------------------------------------------------

// One product's int8 activations [M][K_pad] -> fp16 blocks of `brows` rows x
// one beat (brows * 128 bytes each, swizzled as above), block (mb, kb) at
// xh + (mb * B + kb) * brows * 128, zeros past column K and past row M up to
// mblocks * brows rows.  brows is a multiple of 8 (whole swizzle atoms).
struct CEntry {
    const int8_t *x;       // [M][K_pad]
    uint8_t *xh;           // [mblocks][B][brows * 128 bytes]
    int64_t M;
    int64_t half_begin;    // prefix sum of mblocks*brows*2*B (one thread per row half-beat)
    int32_t K, B;
    int32_t brows, mblocks;
};

struct CList {
    int32_t count;
    int32_t pad_;
    int64_t total;
    CEntry e[TRIT_MAX_LIST_PER_LAUNCH];
};
static_assert(sizeof(CList) <= 32764, "kernel parameter space");

// Fill C.e[i].half_begin and C.total from the other fields and launch the
// conversion (no launch when there is nothing to convert).
cudaError_t launch_act_f16(CList &C, cudaStream_t s);

}  // namespace tc
}  // namespace trit

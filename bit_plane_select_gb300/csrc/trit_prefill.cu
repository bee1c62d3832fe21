// Prefill: y = W x for many activation rows (M >= 64) on the 5th-generation
// tensor cores -- the dense-contraction case of the ternary product.
//
// The product y[m][n] = sum_c x[m][c] * W[n][c] ("Tritium: One Weight Format
// for Ternary Inference ..." -- Introduction, Eq. 3) is contracted by
// tcgen05.mma kind::f16 with fp16 operands and fp32 accumulators in tensor
// memory.  This is exact: int8 activations and +-1 weights are exact in fp16,
// every product is an integer and every partial sum has magnitude <= 128*K <
// 2^24 (the host sends K < 131072 here), so no fp32 addition rounds.  (The
// int8 tensor-core kind is not available on sm_103a.)
//
// Tile: 256 activation rows (two 128-row MMA sub-tiles, two TMEM accumulators
// of 256 columns) x 256 weight rows (MMA N): every expanded weight stage feeds
// both sub-tiles.  One beat of 64 columns per pipeline stage, two operand stages.  Raw inputs (the beat
// of each weight row, the int8 activation halves) arrive kRaw stages ahead by
// 16-byte cp.async copies, each thread copying only what it later converts.
// Warps 0-15 produce each stage:
//   - weights: the beat (pos, neg words) is expanded to 64 fp16 values, two per
//     32-bit word -- (P & m_s) * (0x3C00 >> s) puts +1.0 (0x3C00) in each half
//     whose bit is set (-1.0 = 0xBC00 likewise), m_s = 0x00010001 << s;
//   - activations: int8 -> fp16 by the 1024-bias trick (0x6400 | (x ^ 0x80))
//     minus 1152.
// Both operands use the same column order inside a beat (word k of half h holds
// columns 32h+k and 32h+k+16), so the contraction is unchanged.  Stores go to
// the 128-byte-swizzled K-major layout the MMA descriptors describe.  Warp 16
// issues the MMAs (one thread); the sixteen producer warps then read the
// accumulators (tcgen05.ld), convert to int32 (exact) and write y_i32 / y_f32.
// Every mbarrier wait is bounded: after kWaitNs it sets TRIT_ERR_TIMEOUT and
// the CTA unwinds (waiting, again bounded, for its MMAs before freeing TMEM).
#include "trit_internal.cuh"

namespace trit {
namespace {

constexpr int kBM = 256;                  // activation rows per tile: two 128-row MMA sub-tiles
constexpr int kSubM = 128;                // rows per MMA (TMEM lanes)
constexpr int kBN = 256;                  // weight rows per tile (MMA N)
constexpr int kBK = 64;                   // columns per stage (one beat)
constexpr int kStages = 2;               // MMA operand stages
constexpr int kRaw = 3;                  // raw (plane + int8) copies in flight per producer thread
constexpr int kProducerWarps = 16;
constexpr int kThreads = (kProducerWarps + 1) * 32;
constexpr int kAStage = kBM * kBK * 2;    // 32 KB of fp16 (two 16 KB sub-tiles)
constexpr int kBStage = kBN * kBK * 2;    // 32 KB of fp16
constexpr int kStage = kAStage + kBStage;
constexpr int kRawStage = 2 * kBN * 16 + 2 * (2 * kBM) * 16;   // 512 beats + 512 x-halves x 2 x 16 B
constexpr int kTmemCols = 512;          // two 128 x 256 fp32 accumulators
constexpr int kMaxList = TRIT_MAX_LIST_PER_LAUNCH;
constexpr unsigned long long kWaitNs = 4000000000ull;   // 4 s
constexpr size_t kSmemBytes = size_t(kStages) * kStage + size_t(kRaw) * kRawStage + 1024 + 256;

struct PEntry {
    const uint4 *planes;
    const int8_t *x;        // [M][K_pad]
    const float *x_scale;
    int32_t *y_i32;
    float *y_f32;
    int64_t M, N;
    int64_t tile_begin;     // prefix sum of tiles over the list
    int32_t K, B;
    int32_t mtiles, ntiles;
    float w_scale;
    int32_t pad_;
};

struct PList {
    int32_t count;
    int32_t pad_;
    uint32_t *err;
    int64_t total_tiles;
    PEntry e[kMaxList];
};

// ---- PTX wrappers -------------------------------------------------------------

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
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of the given parity; false after kWaitNs (then *timed_out is set).
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

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, N = 256, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | (uint32_t(kBN >> 3) << 17) |
                            (uint32_t(kSubM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
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

// 1-D bulk copy shared -> global (both 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Barrier among the producer warps only (the MMA warp does not take part).
__device__ __forceinline__ void producers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kProducerWarps * 32) : "memory");
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

// ---- producers -------------------------------------------------------------------

// 16 fp16x2 words (cols 32h + k and 32h + k + 16, k = 0..15) of one plane half.
__device__ __forceinline__ void expand_half(uint32_t P, uint32_t N, uint32_t (&w)[16]) {
    const uint32_t P8 = P >> 8, N8 = N >> 8;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int s = k & 7;
        const uint32_t m = 0x00010001u << s;
        const uint32_t ps = (k < 8 ? P : P8) & m;
        const uint32_t ns = (k < 8 ? N : N8) & m;
        w[k] = ps * (0x3C00u >> s) + ns * (0xBC00u >> s);
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

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PList L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *raw = smem + kStages * kStage;   // kRaw slots of kRawStage bytes
    uint64_t *full = reinterpret_cast<uint64_t *>(raw + kRaw * kRawStage);
    uint64_t *empty = full + kStages;
    uint64_t *done = empty + kStages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    uint32_t *timed_out = tmem_slot + 1;
    uint32_t *viol_any = timed_out + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // tile -> (entry, m tile, n tile)
    int e = 0;
    {
        int a = 0, b = L.count - 1;
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (L.e[mid].tile_begin <= int64_t(blockIdx.x)) a = mid;
            else b = mid - 1;
        }
        e = a;
    }
    const PEntry &E = L.e[e];
    const int64_t tl = int64_t(blockIdx.x) - E.tile_begin;
    const int64_t mt = tl / E.ntiles, nt = tl - mt * E.ntiles;
    const int64_t m0 = mt * kBM, n0 = nt * kBN;
    const int nk = E.B;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], kProducerWarps);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *timed_out = 0;
        *viol_any = 0;
        fence_barrier_init();
    }
    if (warp == kProducerWarps) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kProducerWarps) {
        // thread p: half (p & 1) of weight row n0 + (p >> 1) and half (p & 1) of
        // activation row m0 + (p >> 1) (sub-tile (p >> 1) / 128): equal work per thread
        const int p = threadIdx.x;
        const int hr = p >> 1, hh = p & 1;
        const int64_t wn = n0 + hr;
        const bool w_ok = wn < E.N;
        const uint4 *wrow = E.planes + (w_ok ? wn : 0) * E.B;
        const int ar = hr, ah = hh;
        const int ast = ar / kSubM, arr = ar % kSubM;
        const int64_t xm = m0 + ar;
        const bool x_ok = xm < E.M;
        const int64_t kpad = int64_t(E.B) * 64;
        const uint4 *xrow = reinterpret_cast<const uint4 *>(E.x + (x_ok ? xm : 0) * kpad) + ah * 2;
        uint32_t viol = 0;

        // raw slot layout: [512 beats][512 x-low halves][512 x-high halves], 16 B each
        // (each weight row's beat is copied by both of its threads); every thread
        // copies and later reads only its own pieces
        auto issue = [&](int kb) {
            uint8_t *slot = raw + (kb % kRaw) * kRawStage;
            cp_async16(slot + p * 16, w_ok ? static_cast<const void *>(wrow + kb) : E.planes,
                       w_ok ? 16u : 0u);
            const uint4 *xs = x_ok ? xrow + kb * 4 : reinterpret_cast<const uint4 *>(E.x);
            cp_async16(slot + 2 * kBN * 16 + p * 16, xs, x_ok ? 16u : 0u);
            cp_async16(slot + 2 * kBN * 16 + 2 * kBM * 16 + p * 16, xs + 1, x_ok ? 16u : 0u);
        };
#pragma unroll 1
        for (int r = 0; r < kRaw; ++r) {
            if (r < nk) issue(r);
            cp_async_commit();
        }
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kStages;
            const uint32_t ph = uint32_t(kb / kStages) & 1u;
            cp_async_wait<kRaw - 1>();
            const uint8_t *slot = raw + (kb % kRaw) * kRawStage;
            const uint4 wv = *reinterpret_cast<const uint4 *>(slot + p * 16);
            const uint4 x0 = *reinterpret_cast<const uint4 *>(slot + 2 * kBN * 16 + p * 16);
            const uint4 x1 =
                *reinterpret_cast<const uint4 *>(slot + 2 * kBN * 16 + 2 * kBM * 16 + p * 16);
            if (!mbar_wait(&empty[s], ph ^ 1u, timed_out)) break;
            uint8_t *a_st = smem + s * kStage;
            uint8_t *b_st = a_st + kAStage;
            {   // weights: chunks 4*hh .. 4*hh + 3 of row hr
                viol |= hh ? (wv.y & wv.w) : (wv.x & wv.z);
                uint32_t w[16];
                expand_half(hh ? wv.y : wv.x, hh ? wv.w : wv.z, w);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(b_st + sw128_off(hr, 4 * hh + c)) =
                        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            }
            {   // activations: chunks 4*ah .. 4*ah + 3 of row arr of sub-tile ast
                uint32_t in[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                const int c0 = kb * 64 + ah * 32;
                if (c0 + 32 > E.K) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int lim = E.K - (c0 + 4 * q);   // valid bytes in this word
                        const uint32_t keep = lim >= 4 ? 0xFFFFFFFFu
                                            : (lim <= 0 ? 0u : ((1u << (8 * lim)) - 1u));
                        in[q] &= keep;
                    }
                }
                uint32_t w[16];
                convert_half(in, w);
                uint8_t *a_sub = a_st + ast * (kSubM * kBK * 2);
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(a_sub + sw128_off(arr, 4 * ah + c)) =
                        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
            // the slot's data is consumed (stored above): refill it kRaw stages ahead
            if (kb + kRaw < nk) issue(kb + kRaw);
            cp_async_commit();
        }
        cp_async_wait<0>();
        if (viol) atomicOr(viol_any, 1u);
    } else if (lane == 0) {
        // MMA issue: two 128-row sub-tiles x four K-steps of 16 per stage
        const uint32_t base = smem_u32(smem);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kStages;
            const uint32_t ph = uint32_t(kb / kStages) & 1u;
            if (!mbar_wait(&full[s], ph, timed_out)) break;
            tc_fence_after();
            const uint32_t a_addr = base + s * kStage, b_addr = a_addr + kAStage;
#pragma unroll
            for (int st = 0; st < 2; ++st)
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    mma_f16(tmem + uint32_t(st * kBN),
                            sw128_desc(a_addr + st * (kSubM * kBK * 2) + kk * 32),
                            sw128_desc(b_addr + kk * 32), (kb > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&empty[s]);
        }
        mma_commit(done);   // tracks every MMA issued above
    }

    // epilogue.  For each sub-tile and each output (int32, then fp32): warp w
    // loads TMEM lanes 32*(w%4).. (one activation row per lane) and columns
    // 64*(w/4)..+63, converts, and writes them into a padded row-major staging
    // copy in the freed shared memory; then one 16-byte-aligned bulk copy per
    // row writes it out asynchronously.  Without 16-byte alignment (N % 4 != 0
    // or unaligned outputs) each lane stores its row directly.
    if (warp < kProducerWarps) {
        const bool ok = __all_sync(~0u, mbar_wait(done, 0, timed_out));
        tc_fence_after();
        const bool good = ok && !*reinterpret_cast<volatile uint32_t *>(timed_out);
        const int q = warp & 3, cg = warp >> 2;
        const int p = threadIdx.x;
        const bool bulk = (E.N % 4 == 0) && ((reinterpret_cast<uintptr_t>(E.y_i32) & 15) == 0) &&
                          ((reinterpret_cast<uintptr_t>(E.y_f32) & 15) == 0);
        constexpr int kRowBytes = kBN * 4 + 16;
        const int64_t ncols = E.N - n0 < kBN ? E.N - n0 : kBN;
#pragma unroll 1
        for (int st = 0; st < 2; ++st) {
            const int64_t mrow0 = m0 + st * kSubM;
            if (mrow0 >= E.M) break;
            const int64_t m = mrow0 + 32 * q + lane;
            const bool row_ok = good && m < E.M;
            const float xs = row_ok ? E.x_scale[m] : 0.0f;
#pragma unroll 1
            for (int typ = 0; typ < 2; ++typ) {
                int32_t *yi = typ == 0 ? E.y_i32 : nullptr;
                float *yf = typ == 1 ? E.y_f32 : nullptr;
                if (!yi && !yf) continue;
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    const int col = cg * 64 + half * 32;
                    uint32_t r[32];
                    if (good) {
                        const uint32_t taddr =
                            tmem + (uint32_t(32 * q) << 16) + uint32_t(st * kBN + col);
                        asm volatile(
                            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                            "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,"
                            "%30,%31}, [%32];"
                            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                              "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                              "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
                              "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                              "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]),
                              "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                            : "r"(taddr));
                        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                    }
                    uint32_t v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int32_t y = __float2int_rn(__uint_as_float(r[i]));
                        v[i] = yi ? uint32_t(y) : __float_as_uint(dequant(y, E.w_scale, xs));
                    }
                    if (bulk) {
                        uint8_t *dst = smem + (32 * q + lane) * kRowBytes + col * 4;
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<uint4 *>(dst + i * 4) =
                                make_uint4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                    } else if (row_ok) {
                        uint32_t *o = yi ? reinterpret_cast<uint32_t *>(yi)
                                         : reinterpret_cast<uint32_t *>(yf);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (n0 + col + i < E.N) o[m * E.N + n0 + col + i] = v[i];
                    }
                }
                if (bulk) {
                    fence_proxy_async();
                    producers_sync();
                    if (good && p < kSubM && mrow0 + p < E.M) {
                        uint8_t *g = yi ? reinterpret_cast<uint8_t *>(yi) : reinterpret_cast<uint8_t *>(yf);
                        bulk_store(g + ((mrow0 + p) * E.N + n0) * 4, smem + p * kRowBytes,
                                   uint32_t(ncols * 4));
                        bulk_commit();
                        bulk_wait_read();   // the staging rows may be rewritten after this
                    }
                    producers_sync();
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        uint32_t f = 0;
        if (*timed_out) f |= TRIT_ERR_TIMEOUT;
        if (*viol_any) f |= TRIT_ERR_P1;
        if (f) atomicOr(L.err, f);
    }
    if (warp == kProducerWarps)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

}  // namespace

bool prefill_supported(const ProjDev &p) {
    return p.M >= kPrefillMinM && p.K < 131072;
}

cudaError_t launch_prefill_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s) {
    static thread_local PList L;
    cudaError_t ae = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          int(kSmemBytes));
    if (ae != cudaSuccess) return ae;
    for (int base = 0; base < count; base += kMaxList) {
        const int n = count - base < kMaxList ? count - base : kMaxList;
        L.count = n;
        L.pad_ = 0;
        L.err = err;
        int64_t tiles = 0;
        for (int i = 0; i < n; ++i) {
            const ProjDev &p = list[base + i];
            PEntry &E = L.e[i];
            E.planes = p.planes;
            E.x = p.x;
            E.x_scale = p.x_scale;
            E.y_i32 = p.y_i32;
            E.y_f32 = p.y_f32;
            E.M = p.M;
            E.N = p.N;
            E.K = p.K;
            E.B = p.B;
            E.mtiles = int32_t((p.M + kBM - 1) / kBM);
            E.ntiles = int32_t((p.N + kBN - 1) / kBN);
            E.w_scale = p.w_scale;
            E.pad_ = 0;
            E.tile_begin = tiles;
            tiles += int64_t(E.mtiles) * E.ntiles;
        }
        L.total_tiles = tiles;
        prefill_kernel<<<dim3(unsigned(tiles)), kThreads, kSmemBytes, s>>>(L);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace trit

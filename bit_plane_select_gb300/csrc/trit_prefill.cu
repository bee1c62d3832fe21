// Prefill: y = W x for many activation rows (M >= 17) on the 5th-generation
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
// Two launches per list of products:
//  1. act_f16_kernel converts each product's int8 activations once into a
//     temporary fp16 copy laid out as 16 KB blocks of 128 rows x one beat (64
//     columns), each block already in the MMA's 128-byte-swizzled K-major
//     order, with columns permuted inside the beat (word k of half h holds
//     columns 32h+k and 32h+k+16) and zeros past column K and past row M.
//  2. prefill_kernel: tile = 256 activation rows (two 128-row MMA sub-tiles,
//     two TMEM accumulators of 128 columns) x 128 weight rows (MMA N); one
//     beat per pipeline stage, two stages.  Per stage one thread brings the
//     two activation blocks with bulk copies that complete on the stage's
//     mbarrier; eight producer warps (two threads per weight row, half a beat
//     each) expand the 128 weight beats to fp16 +-1 in the same column order
//     ((P & m_s) * (0x3C00 >> s) sets +1.0 in each half whose bit is set, -1.0 =
//     0xBC00 likewise), so each expanded beat feeds both sub-tiles.  One thread
//     of warp 8 issues the MMAs; the producer warps then read the fp32
//     accumulators (exact integers), convert, and write them through a per-warp
//     transpose in the freed shared memory so that stores cover whole row
//     segments.  Two CTAs share an SM (256 tensor-memory columns and ~106 KB of
//     shared memory each), so one CTA's epilogue runs while the other's MMAs do.
// The fp16 copy of the activations is scratch memory: the host allocates it
// stream-ordered around the two launches.
// Every mbarrier wait is bounded: after kWaitNs it sets TRIT_ERR_TIMEOUT and
// the CTA unwinds (waiting, again bounded, for its MMAs before freeing TMEM).
#include "trit_internal.cuh"

namespace trit {
namespace {

constexpr int kSubM = 128;                // rows per MMA (TMEM lanes)
constexpr int kSubs = 2;                  // MMA sub-tiles per tile
constexpr int kBM = kSubM * kSubs;        // activation rows per tile
constexpr int kBN = 128;                  // weight rows per tile (MMA N)
constexpr int kBK = 64;                   // columns per stage (one beat)
constexpr int kStages = 2;                // MMA operand stages
constexpr int kRaw = 4;                   // plane half-beats in flight per producer thread
constexpr int kProducerWarps = 8;
constexpr int kThreads = (kProducerWarps + 1) * 32;
constexpr int kBlock = kSubM * kBK * 2;   // one 16 KB activation block (fp16)
constexpr int kAStage = kSubs * kBlock;   // 32 KB
constexpr int kBStage = kBN * kBK * 2;    // 16 KB
constexpr int kStage = kAStage + kBStage;
constexpr int kRawStage = kProducerWarps * 32 * 8;    // per thread: its half of pos and neg
constexpr int kTmemCols = kSubs * kBN;    // 256: two 128 x 128 fp32 accumulators
constexpr int kMaxList = TRIT_MAX_LIST_PER_LAUNCH;
constexpr unsigned long long kWaitNs = 4000000000ull;   // 4 s
constexpr size_t kSmemBytes = size_t(kStages) * kStage + size_t(kRaw) * kRawStage + 1024 + 256;
static_assert(kProducerWarps * 32 == 2 * kBN, "two producer threads per weight beat");
// two CTAs share an SM (tensor memory 2 x 256 columns, shared memory 2 x ~106 KB),
// so one CTA's epilogue overlaps the other's MMAs
constexpr int kCtasPerSm = 2;
static_assert(kCtasPerSm * kTmemCols <= 512, "tensor memory of the resident CTAs");

struct PEntry {
    const uint4 *planes;
    const uint8_t *xh;      // blocked fp16 activations: [mblocks][B][kBlock bytes]
    const float *x_scale;
    int32_t *y_i32;
    float *y_f32;
    int64_t M, N;
    int64_t tile_begin;     // prefix sum of tiles over the list
    int32_t K, B;
    int32_t mtiles, ntiles;
    int32_t mblocks;        // ceil(M / 128)
    float w_scale;
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
// K-major, N = 128, M = 128.
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
// 4-byte asynchronous global -> shared copy; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async4(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
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

// ---- producers -------------------------------------------------------------------

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

// ---- activation conversion: int8 [M][K_pad] -> blocked, swizzled fp16 -------------

struct CEntry {
    const int8_t *x;       // [M][K_pad]
    uint8_t *xh;           // [mblocks][B][kBlock bytes]
    int64_t M;
    int64_t half_begin;    // prefix sum of mblocks*128*2*B (one thread per row half-beat)
    int32_t K, B;
};

struct CList {
    int32_t count;
    int32_t pad_;
    int64_t total;
    CEntry e[kMaxList];
};

// One thread per (row, half-beat): 32 int8 in, 4 fp16 chunks of 16 bytes out.
__global__ void __launch_bounds__(256) act_f16_kernel(const __grid_constant__ CList L) {
    for (int64_t g = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; g < L.total;
         g += int64_t(gridDim.x) * blockDim.x) {
        int a = 0, b = L.count - 1;
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (L.e[mid].half_begin <= g) a = mid;
            else b = mid - 1;
        }
        const CEntry &E = L.e[a];
        const int64_t i = g - E.half_begin;
        const int64_t halves_per_row = 2 * int64_t(E.B);
        const int64_t m = i / halves_per_row;
        const int hb = int(i - m * halves_per_row);     // half-beat index along the row
        const int kb = hb >> 1, h = hb & 1;
        uint32_t in[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        const int c0 = hb * 32;
        if (m < E.M) {
            const uint4 *src = reinterpret_cast<const uint4 *>(E.x + m * (int64_t(E.B) * 64) + c0);
            const uint4 u0 = src[0], u1 = src[1];
            in[0] = u0.x; in[1] = u0.y; in[2] = u0.z; in[3] = u0.w;
            in[4] = u1.x; in[5] = u1.y; in[6] = u1.z; in[7] = u1.w;
            if (c0 + 32 > E.K) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int lim = E.K - (c0 + 4 * q);
                    const uint32_t keep = lim >= 4 ? 0xFFFFFFFFu : (lim <= 0 ? 0u : ((1u << (8 * lim)) - 1u));
                    in[q] &= keep;
                }
            }
        }
        uint32_t w[16];
        convert_half(in, w);   // rows past M hold x = 0 and convert to +0.0
        const int r = int(m % kSubM);
        uint8_t *blk = E.xh + ((m / kSubM) * E.B + kb) * int64_t(kBlock);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4 *>(blk + sw128_off(r, 4 * h + c)) =
                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}

// ---- the tensor-core product ---------------------------------------------------------

__global__ void __launch_bounds__(kThreads, kCtasPerSm) prefill_kernel(const __grid_constant__ PList L) {
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
    const int nsub = int(E.mblocks - mt * kSubs < kSubs ? E.mblocks - mt * kSubs : kSubs);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], kProducerWarps + 1);   // 16 warps + the expect_tx arrival
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
        // thread p: half (p & 1) of weight row n0 + (p >> 1)
        const int p = threadIdx.x;
        const int br = p >> 1, bh = p & 1;
        const int64_t wn = n0 + br;
        const bool w_ok = wn < E.N;
        const uint8_t *wrow = reinterpret_cast<const uint8_t *>(E.planes + (w_ok ? wn : 0) * E.B);
        const uint8_t *xblk = E.xh + (mt * kSubs) * int64_t(E.B) * kBlock;   // block (mt*kSubs, 0)
        uint32_t viol = 0;
        auto issue = [&](int kb) {   // this half's pos word and neg word of beat kb
            uint8_t *slot = raw + (kb % kRaw) * kRawStage + p * 8;
            const uint8_t *beat = wrow + int64_t(kb) * 16;
            cp_async4(slot, beat + 4 * bh, w_ok ? 4u : 0u);
            cp_async4(slot + 4, beat + 8 + 4 * bh, w_ok ? 4u : 0u);
        };
#pragma unroll 1
        for (int r = 0; r < kRaw; ++r) {
            if (r < nk) issue(r);
            cp_async_commit();
        }
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kStages;
            const uint32_t ph = uint32_t(kb / kStages) & 1u;
            if (!mbar_wait(&empty[s], ph ^ 1u, timed_out)) break;
            uint8_t *a_st = smem + s * kStage;
            uint8_t *b_st = a_st + kAStage;
            if (p == 0) {   // the activation blocks of this stage
                mbar_arrive_expect_tx(&full[s], uint32_t(nsub) * kBlock);
                for (int st = 0; st < nsub; ++st)
                    bulk_load(a_st + st * kBlock, xblk + (int64_t(st) * E.B + kb) * kBlock, kBlock,
                              &full[s]);
            }
            cp_async_wait<kRaw - 1>();
            const uint2 pn = *reinterpret_cast<const uint2 *>(raw + (kb % kRaw) * kRawStage + p * 8);
            viol |= pn.x & pn.y;
            {   // weights: chunks 4*bh .. 4*bh+3 of row br
                uint32_t w[8];
                expand_quarter(pn.x, pn.y, w);
                *reinterpret_cast<uint4 *>(b_st + sw128_off(br, 4 * bh)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(b_st + sw128_off(br, 4 * bh + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
                expand_quarter(pn.x >> 8, pn.y >> 8, w);
                *reinterpret_cast<uint4 *>(b_st + sw128_off(br, 4 * bh + 2)) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4 *>(b_st + sw128_off(br, 4 * bh + 3)) = make_uint4(w[4], w[5], w[6], w[7]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[s]);
            // the raw slot is consumed: refill it kRaw stages ahead
            if (kb + kRaw < nk) issue(kb + kRaw);
            cp_async_commit();
        }
        cp_async_wait<0>();
        if (viol) atomicOr(viol_any, 1u);
    } else if (lane == 0) {
        // MMA issue: up to four 128-row sub-tiles x four K-steps of 16 per stage
        const uint32_t base = smem_u32(smem);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % kStages;
            const uint32_t ph = uint32_t(kb / kStages) & 1u;
            if (!mbar_wait(&full[s], ph, timed_out)) break;
            tc_fence_after();
            const uint32_t a_addr = base + s * kStage, b_addr = a_addr + kAStage;
            for (int st = 0; st < nsub; ++st)
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    mma_f16(tmem + uint32_t(st * kBN), sw128_desc(a_addr + st * kBlock + kk * 32),
                            sw128_desc(b_addr + kk * 32), (kb > 0 || kk > 0) ? 1u : 0u);
            mma_commit(&empty[s]);
        }
        mma_commit(done);   // tracks every MMA issued above
    }

    // epilogue.  For each sub-tile: warp w loads TMEM lanes 32*(w%4).. (one
    // activation row per lane) and columns 32*(w/4)..+31; for each output
    // (int32, then fp32) the lanes write their rows into the warp's own padded
    // 32 x 32 staging tile in the freed shared memory and read it back
    // transposed, so every store instruction writes whole 128-byte row
    // segments (16-byte vectors when the rows are 16-byte aligned).
    if (warp < kProducerWarps) {
        const bool ok = __all_sync(~0u, mbar_wait(done, 0, timed_out));
        tc_fence_after();
        const bool good = ok && !*reinterpret_cast<volatile uint32_t *>(timed_out);
        const int q = warp & 3;
        const bool vec = (E.N % 4 == 0) && ((reinterpret_cast<uintptr_t>(E.y_i32) & 15) == 0) &&
                         ((reinterpret_cast<uintptr_t>(E.y_f32) & 15) == 0);
        constexpr int kPitch = 36;   // words per staging row: 32 + 4 of padding
        uint32_t *sw = reinterpret_cast<uint32_t *>(smem) + warp * (32 * kPitch);
#pragma unroll 1
        for (int sc = 0; sc < nsub * 2; ++sc) {   // (sub-tile, column group) pairs of this warp
            const int st = sc >> 1;
            const int cg = (warp >> 2) + 2 * (sc & 1);
            const int col = cg * 32;
            const int64_t mbase = m0 + st * kSubM + 32 * q;   // rows of this warp
            const int64_t m = mbase + lane;
            const float xs = (good && m < E.M) ? E.x_scale[m] : 0.0f;
            uint32_t r[32];
            if (good) {
                const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(st * kBN + col);
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
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = 0;
            }
            if (!good) continue;
#pragma unroll 1
            for (int typ = 0; typ < 2; ++typ) {
                uint32_t *out = typ == 0 ? reinterpret_cast<uint32_t *>(E.y_i32)
                                         : reinterpret_cast<uint32_t *>(E.y_f32);
                if (!out) continue;
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    uint32_t v[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int32_t y = __float2int_rn(__uint_as_float(r[i + k]));
                        v[k] = typ == 0 ? uint32_t(y) : __float_as_uint(dequant(y, E.w_scale, xs));
                    }
                    *reinterpret_cast<uint4 *>(sw + lane * kPitch + i) = make_uint4(v[0], v[1], v[2], v[3]);
                }
                __syncwarp();
                if (vec) {
#pragma unroll
                    for (int it = 0; it < 8; ++it) {
                        const int rr = it * 4 + (lane >> 3), c4 = (lane & 7) * 4;
                        const int64_t mm = mbase + rr, n = n0 + col + c4;
                        const uint4 val = *reinterpret_cast<const uint4 *>(sw + rr * kPitch + c4);
                        if (mm < E.M && n < E.N)
                            *reinterpret_cast<uint4 *>(out + mm * E.N + n) = val;
                    }
                } else {
#pragma unroll 4
                    for (int rr = 0; rr < 32; ++rr) {
                        const int64_t mm = mbase + rr, n = n0 + col + lane;
                        if (mm < E.M && n < E.N) out[mm * E.N + n] = sw[rr * kPitch + lane];
                    }
                }
                __syncwarp();
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

// Bytes of the blocked fp16 activation copy of one product.
int64_t act_f16_bytes(const ProjDev &p) {
    return ((p.M + kSubM - 1) / kSubM) * int64_t(p.B) * kBlock;
}

// Convert and multiply the products list[0..n) with their fp16 activation
// copies at xh[i] (each act_f16_bytes long, 16-byte aligned).
cudaError_t launch_two(const ProjDev *list, int n, uint8_t *const *xh, uint32_t *err, cudaStream_t s) {
    static thread_local CList C;
    static thread_local PList L;
    C.count = n;
    C.pad_ = 0;
    L.count = n;
    L.pad_ = 0;
    L.err = err;
    int64_t halves = 0, tiles = 0;
    for (int i = 0; i < n; ++i) {
        const ProjDev &p = list[i];
        const int64_t mblocks = (p.M + kSubM - 1) / kSubM;
        CEntry &c = C.e[i];
        c.x = p.x;
        c.xh = xh[i];
        c.M = p.M;
        c.K = p.K;
        c.B = p.B;
        c.half_begin = halves;
        halves += mblocks * kSubM * 2 * int64_t(p.B);
        PEntry &E = L.e[i];
        E.planes = p.planes;
        E.xh = xh[i];
        E.x_scale = p.x_scale;
        E.y_i32 = p.y_i32;
        E.y_f32 = p.y_f32;
        E.M = p.M;
        E.N = p.N;
        E.K = p.K;
        E.B = p.B;
        E.mblocks = int32_t(mblocks);
        E.mtiles = int32_t((p.M + kBM - 1) / kBM);
        E.ntiles = int32_t((p.N + kBN - 1) / kBN);
        E.w_scale = p.w_scale;
        E.tile_begin = tiles;
        tiles += int64_t(E.mtiles) * E.ntiles;
    }
    C.total = halves;
    L.total_tiles = tiles;
    int64_t cblocks = (halves + 255) / 256;
    const int64_t cap = int64_t(device_sm_count()) * 16;
    cblocks = cblocks < cap ? cblocks : cap;
    act_f16_kernel<<<int(cblocks), 256, 0, s>>>(C);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    prefill_kernel<<<dim3(unsigned(tiles)), kThreads, kSmemBytes, s>>>(L);
    return cudaGetLastError();
}

}  // namespace

bool prefill_supported(const ProjDev &p) {
    return p.M >= kPrefillMinM && p.K < 131072;
}

int64_t prefill_scratch_bytes(const ProjDev &p) { return act_f16_bytes(p); }

cudaError_t launch_prefill_into(const ProjDev &p, uint8_t *xh, uint32_t *err, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kSmemBytes));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    uint8_t *const one[1] = {xh};
    return launch_two(&p, 1, one, err, s);
}

// The fp16 activation copies are allocated stream-ordered (cudaMallocAsync on
// `s`) and freed after the launches, in groups of at most kScratchGroup bytes.
cudaError_t launch_prefill_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s) {
    constexpr int64_t kScratchGroup = int64_t(1) << 30;
    cudaError_t ae = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          int(kSmemBytes));
    if (ae != cudaSuccess) return ae;
    ae = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (ae != cudaSuccess) return ae;
    static thread_local uint8_t *xh[kMaxList];
    int base = 0;
    while (base < count) {
        int n = 0;
        int64_t bytes = 0;
        while (base + n < count && n < kMaxList) {
            const int64_t b = (act_f16_bytes(list[base + n]) + 255) & ~int64_t(255);
            if (n > 0 && bytes + b > kScratchGroup) break;
            bytes += b;
            ++n;
        }
        uint8_t *buf = nullptr;
        cudaError_t e = cudaMallocAsync(reinterpret_cast<void **>(&buf), size_t(bytes), s);
        if (e != cudaSuccess) return e;
        int64_t off = 0;
        for (int i = 0; i < n; ++i) {
            xh[i] = buf + off;
            off += (act_f16_bytes(list[base + i]) + 255) & ~int64_t(255);
        }
        e = launch_two(list + base, n, xh, err, s);
        cudaError_t f = cudaFreeAsync(buf, s);
        if (e != cudaSuccess) return e;
        if (f != cudaSuccess) return f;
        base += n;
    }
    return cudaSuccess;
}

}  // namespace trit

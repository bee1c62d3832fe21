// Prefill: y = W x for many activation rows (M > 128) on the 5th-generation
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
//     columns 32h+k and 32h+k+16) and zeros past column K and past row M (the
//     row blocks are padded to an even count).
//  2. prefill_kernel: persistent, one CTA pair (a cluster of two CTAs on two
//     SMs) per pair tile of 256 activation rows x 256 weight rows.  The pair
//     issues tcgen05.mma.cta_group::2 with M = 256, N = 256: CTA r holds
//     activation rows 128r.. of the tile (operand A) and expands weight rows
//     128r.. of the tile (its half of operand B); its tensor memory receives
//     its 128 rows x all 256 columns.  One beat per pipeline stage, five stages
//     of 32 KB per CTA.  Per stage one thread brings the CTA's activation block
//     with a bulk copy; four producer warps (one thread per weight row: its
//     beat arrives by a 16-byte cp.async) expand the 128 weight beats to fp16
//     +-1 in the same column
//     order ((P & m_s) * (0x3C00 >> s) sets +1.0 in each half whose bit is
//     set, -1.0 = 0xBC00 likewise).  In the leader CTA (rank 0) one thread
//     issues the MMAs once both CTAs' stages are full (the peer's MMA warp
//     relays its CTA's stage completion to the leader's barrier) and commits
//     to barriers in both CTAs.  Two 256-column accumulators alternate between
//     tiles, so eight epilogue warps per CTA read one tile's accumulator
//     (exact integers), convert, and write it through a per-warp transpose in
//     shared memory (whole 128-byte row segments per store) while the MMAs of
//     the next tile run.
// Per SM this takes N = 256 MMAs (each SM computes 128 x 256 per instruction)
// with 128 expanded weight rows per 256 activation rows of the pair, and reads
// each activation block once per 256 weight rows.
// The fp16 copy of the activations is scratch memory: the host allocates it
// stream-ordered around the two launches.
// Every mbarrier wait is bounded: after kWaitNs it sets TRIT_ERR_TIMEOUT and
// the roles unwind; before tensor memory is freed each CTA waits, again
// bounded, for the last MMA commit.
#include "trit_tc.cuh"

namespace trit {
namespace {

using namespace tc;

constexpr int kSubM = 128;                // activation rows per CTA (TMEM lanes)
constexpr int kPairM = 2 * kSubM;         // activation rows per pair tile (MMA M)
constexpr int kHalfN = 128;               // weight rows expanded per CTA
constexpr int kPairN = 2 * kHalfN;        // weight rows per pair tile (MMA N)
constexpr int kStages = 5;                // MMA operand stages
constexpr int kRaw = 4;                   // plane half-beats in flight per producer thread
constexpr int kProducerWarps = 4;   // measured: 2 / 8 / 16 warps are slower (the
                                    // per-thread proxy fence of each stage is the cost)
constexpr int kMmaWarp = kProducerWarps;  // MMA issue (leader) or relay (peer)
constexpr int kEpiWarp0 = kMmaWarp + 1;
constexpr int kEpiWarps = 8;              // two per TMEM lane quarter, 128 columns each
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr int kBlock = kSubM * kBK * 2;   // one 16 KB activation block (fp16)
constexpr int kBStage = kHalfN * kBK * 2; // 16 KB of expanded weights
constexpr int kStage = kBlock + kBStage;
constexpr int kRawStage = kProducerWarps * 32 * 16;   // per thread: its row's beat
constexpr int kAccCols = kPairN;          // fp32 columns of one accumulator
constexpr int kTmemCols = 2 * kAccCols;   // two accumulators: all 512 columns
constexpr int kPitch = 36;                // words per epilogue staging row: 32 + 4 of padding
constexpr int kEpiBytes = kEpiWarps * 32 * kPitch * 4;
constexpr int kMaxList = TRIT_MAX_LIST_PER_LAUNCH;
constexpr size_t kSmemBytes = 1024 + size_t(kStages) * kStage + size_t(kRaw) * kRawStage +
                              kEpiBytes + 256;
static_assert(kProducerWarps * 32 == kHalfN, "one producer thread per weight beat");
static_assert(kSmemBytes <= 227 * 1024, "shared memory of one CTA");

struct PEntry {
    const uint4 *planes;
    const uint8_t *xh;      // blocked fp16 activations: [mblocks][B][kBlock bytes]
    const float *x_scale;
    int32_t *y_i32;
    float *y_f32;
    int64_t M, N;
    int64_t tile_begin;     // prefix sum of pair tiles over the list
    int32_t K, B;
    int32_t mtiles, ntiles; // pair tiles along M (256 rows) and N (256 rows)
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
static_assert(sizeof(PList) <= 32764, "kernel parameter space");


// ---- pair-specific PTX wrappers (the shared ones are in trit_tc.cuh) ---------

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, N = 256, M = 256 (the pair).
constexpr uint32_t kIdesc = (1u << 4) | (0u << 7) | (0u << 10) | (uint32_t(kPairN >> 3) << 17) |
                            (uint32_t(kPairM >> 4) << 24);

__device__ __forceinline__ void mma_pair(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate));
}

// Arrive on the barrier at the same offset in both CTAs of the pair once every
// MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(smem_u32(bar)),
        "h"(uint16_t(3))
        : "memory");
}

// Arrive (release, cluster scope) on the barrier at the same offset in CTA `rank`.
__device__ __forceinline__ void mbar_arrive_at(uint64_t *bar, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}

// The same arrive without release semantics.  Measured: a cluster-scope release
// costs the issuing SM about 0.7 us and does not overlap with others, so the
// per-stage relay uses this form.  It is issued only after the relaying thread
// has observed (acquire) the completion of its own CTA's stage barrier -- the
// bulk copy's bytes and the producer warps' stores (each fenced to the async
// proxy and released at CTA scope) are then in that CTA's shared memory, which
// the leader's MMA reads directly.
__device__ __forceinline__ void mbar_arrive_at_relaxed(uint64_t *bar, uint32_t rank) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(bar)), "r"(rank));
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}


// ---- activation conversion: int8 [M][K_pad] -> blocked, swizzled fp16 -------------

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
        const int64_t br = E.brows;
        const int r = int(m % br);
        uint8_t *blk = E.xh + ((m / br) * E.B + kb) * (br * 128);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            *reinterpret_cast<uint4 *>(blk + sw128_off(r, 4 * h + c)) =
                make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
    }
}


// ---- the tensor-core product ---------------------------------------------------------

// Pair tile t -> entry, m tile, n tile.
struct TileRef {
    int e;
    int64_t mt, nt;
};
__device__ __forceinline__ TileRef tile_ref(const PList &L, int64_t t) {
    int a = 0, b = L.count - 1;
    while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (L.e[mid].tile_begin <= t) a = mid;
        else b = mid - 1;
    }
    TileRef r;
    r.e = a;
    const int64_t tl = t - L.e[a].tile_begin;
    r.mt = tl / L.e[a].ntiles;
    r.nt = tl - r.mt * L.e[a].ntiles;
    return r;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ PList L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *raw = smem + kStages * kStage;            // kRaw slots of kRawStage bytes
    uint32_t *epi = reinterpret_cast<uint32_t *>(raw + kRaw * kRawStage);
    uint64_t *full = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(epi) + kEpiBytes);
    uint64_t *empty = full + kStages;
    uint64_t *tfull = empty + kStages;      // accumulator a holds a finished tile
    uint64_t *tempty = tfull + 2;           // accumulator a has been read (leader's counts)
    uint64_t *done = tempty + 2;            // every MMA has completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    uint32_t *timed_out = tmem_slot + 1;
    uint32_t *viol_any = timed_out + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int64_t pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            // producer warps + the expect_tx arrival (+ the peer's relay in the leader)
            mbar_init(&full[s], kProducerWarps + 1 + (rank == 0 ? 1 : 0));
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * kEpiWarps);
        }
        mbar_init(done, 1);
        *timed_out = 0;
        *viol_any = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    tc_fence_before();
    cluster_sync_all();   // both CTAs' barriers exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kProducerWarps) {
        // thread p: weight row 128*rank + p of each tile, the whole beat
        const int p = threadIdx.x;
        const int br = p;
        // load cursor (kRaw stages ahead of the consume cursor, across tiles)
        int64_t lt = pair;
        int lkb = 0, lnk = 0;
        const uint8_t *lrow = nullptr;
        uint32_t lbytes = 0;
        auto load_tile = [&](int64_t t) {
            const TileRef r = tile_ref(L, t);
            const PEntry &E = L.e[r.e];
            const int64_t wn = r.nt * kPairN + int64_t(rank) * kHalfN + br;
            const bool ok = wn < E.N;
            lrow = reinterpret_cast<const uint8_t *>(E.planes + (ok ? wn : 0) * E.B);
            lbytes = ok ? 16u : 0u;
            lnk = E.B;
            lkb = 0;
        };
        if (lt < L.total_tiles) load_tile(lt);
        int64_t li = 0;   // loads issued
        auto issue_next = [&]() {   // the row's next beat (pos and neg words)
            if (lt < L.total_tiles) {
                uint8_t *slot = raw + int(li % kRaw) * kRawStage + p * 16;
                const uint8_t *beat = lrow + int64_t(lkb) * 16;
                cp_async16(slot, beat, lbytes);
                ++li;
                if (++lkb == lnk) {
                    lt += npairs;
                    if (lt < L.total_tiles) load_tile(lt);
                }
            }
            cp_async_commit();
        };
#pragma unroll 1
        for (int r = 0; r < kRaw; ++r) issue_next();
        uint32_t viol = 0;
        int64_t it = 0;   // stages consumed
        bool stop = false;
        for (int64_t t = pair; t < L.total_tiles && !stop; t += npairs) {
            const TileRef r = tile_ref(L, t);
            const PEntry &E = L.e[r.e];
            const int nk = E.B;
            const uint8_t *xblk = E.xh + (2 * r.mt + rank) * int64_t(E.B) * kBlock;
            for (int kb = 0; kb < nk; ++kb, ++it) {
                const int s = int(it % kStages);
                const uint32_t ph = uint32_t(it / kStages) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, timed_out)) {
                    stop = true;
                    break;
                }
                uint8_t *a_st = smem + s * kStage;
                uint8_t *b_st = a_st + kBlock;
                if (p == 0) {   // the activation block of this stage
                    mbar_arrive_expect_tx(&full[s], kBlock);
                    bulk_load(a_st, xblk + int64_t(kb) * kBlock, kBlock, &full[s]);
                }
                cp_async_wait<kRaw - 1>();
                const uint4 pn = *reinterpret_cast<const uint4 *>(raw + int(it % kRaw) * kRawStage + p * 16);
                viol |= (pn.x & pn.z) | (pn.y & pn.w);
#pragma unroll
                for (int bh = 0; bh < 2; ++bh) {   // weights: chunks 4*bh .. 4*bh+3 of row br
                    const uint32_t P = bh ? pn.y : pn.x, Q = bh ? pn.w : pn.z;
                    uint32_t w[8];
                    expand_quarter(P, Q, w);
                    *reinterpret_cast<uint4 *>(b_st + sw128_off(br, 4 * bh)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(b_st + sw128_off(br, 4 * bh + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
                    expand_quarter(P >> 8, Q >> 8, w);
                    *reinterpret_cast<uint4 *>(b_st + sw128_off(br, 4 * bh + 2)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(b_st + sw128_off(br, 4 * bh + 3)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[s]);
                issue_next();   // the raw slot is consumed: refill it kRaw stages ahead
            }
        }
        cp_async_wait<0>();
        if (viol) atomicOr(viol_any, 1u);
    } else if (warp == kMmaWarp) {
        if (lane == 0 && rank == 0) {
            // MMA issue: per stage four K-steps of 16 into the tile's accumulator
            const uint32_t base = smem_u32(smem);
            int64_t it = 0, i = 0;
            bool stop = false;
            for (int64_t t = pair; t < L.total_tiles && !stop; t += npairs, ++i) {
                const int a = int(i & 1);
                const uint32_t use = uint32_t(i >> 1);
                if (!mbar_wait(&tempty[a], (use & 1u) ^ 1u, timed_out)) break;
                tc_fence_after();
                const int nk = L.e[tile_ref(L, t).e].B;
                const uint32_t d = tmem + uint32_t(a * kAccCols);
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = int(it % kStages);
                    const uint32_t ph = uint32_t(it / kStages) & 1u;
                    if (!mbar_wait(&full[s], ph, timed_out)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = base + s * kStage, b_addr = a_addr + kBlock;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_pair(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32),
                                 (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit_pair(&empty[s]);
                }
                if (!stop) mma_commit_pair(&tfull[a]);
            }
            mma_commit_pair(done);   // tracks every MMA issued above
        } else if (lane == 0) {
            // peer: relay each full stage of this CTA to the leader's barrier
            int64_t it = 0;
            bool stop = false;
            for (int64_t t = pair; t < L.total_tiles && !stop; t += npairs) {
                const int nk = L.e[tile_ref(L, t).e].B;
                for (int kb = 0; kb < nk; ++kb, ++it) {
                    const int s = int(it % kStages);
                    const uint32_t ph = uint32_t(it / kStages) & 1u;
                    if (!mbar_wait(&full[s], ph, timed_out)) {
                        stop = true;
                        break;
                    }
                    mbar_arrive_at_relaxed(&full[s], 0);
                }
            }
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads TMEM lanes 32*(w%4).. (one activation row per
        // lane) and columns 128*h .. 128*h+127 (h = which of the two warps of
        // that lane quarter) and, 32 columns at a time, passes the int32 sums
        // through its padded 32 x 32 staging tile, read back transposed so every
        // store (int32, and the fp32 dequantisation computed from the same
        // read) writes whole 128-byte row segments.
        const int q = warp & 3;
        const int h = (warp - kEpiWarp0) >> 2;
        uint32_t *sw = epi + (warp - kEpiWarp0) * (32 * kPitch);
        int64_t i = 0;
        for (int64_t t = pair; t < L.total_tiles; t += npairs, ++i) {
            const int a = int(i & 1);
            const uint32_t use = uint32_t(i >> 1);
            const bool ok = __all_sync(~0u, mbar_wait(&tfull[a], use & 1u, timed_out));
            if (!ok) break;
            tc_fence_after();
            const TileRef r = tile_ref(L, t);
            const PEntry &E = L.e[r.e];
            const bool vec = (E.N % 4 == 0) && ((reinterpret_cast<uintptr_t>(E.y_i32) & 15) == 0) &&
                             ((reinterpret_cast<uintptr_t>(E.y_f32) & 15) == 0);
            const int64_t mbase = r.mt * kPairM + int64_t(rank) * kSubM + 32 * q;   // rows of this warp
            const int64_t m = mbase + lane;
            const float xs = m < E.M ? E.x_scale[m] : 0.0f;
            const int64_t n0 = r.nt * kPairN;
#pragma unroll 1
            for (int cg = 0; cg < kAccCols / 64; ++cg) {
                const int col = h * (kAccCols / 2) + cg * 32;
                uint32_t v32[32];
                const uint32_t taddr = tmem + (uint32_t(32 * q) << 16) + uint32_t(a * kAccCols + col);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                    "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,"
                    "%30,%31}, [%32];"
                    : "=r"(v32[0]), "=r"(v32[1]), "=r"(v32[2]), "=r"(v32[3]), "=r"(v32[4]),
                      "=r"(v32[5]), "=r"(v32[6]), "=r"(v32[7]), "=r"(v32[8]), "=r"(v32[9]),
                      "=r"(v32[10]), "=r"(v32[11]), "=r"(v32[12]), "=r"(v32[13]), "=r"(v32[14]),
                      "=r"(v32[15]), "=r"(v32[16]), "=r"(v32[17]), "=r"(v32[18]), "=r"(v32[19]),
                      "=r"(v32[20]), "=r"(v32[21]), "=r"(v32[22]), "=r"(v32[23]), "=r"(v32[24]),
                      "=r"(v32[25]), "=r"(v32[26]), "=r"(v32[27]), "=r"(v32[28]), "=r"(v32[29]),
                      "=r"(v32[30]), "=r"(v32[31])
                    : "r"(taddr));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (n0 + col >= E.N) continue;   // past the last weight row
                // the int32 values into this lane's staging row, read back transposed;
                // each value read back is stored as int32 and, dequantised with its
                // row's scale (from the lane that holds that row), as fp32
#pragma unroll
                for (int c = 0; c < 32; c += 4)
                    *reinterpret_cast<uint4 *>(sw + lane * kPitch + c) = make_uint4(
                        uint32_t(__float2int_rn(__uint_as_float(v32[c]))),
                        uint32_t(__float2int_rn(__uint_as_float(v32[c + 1]))),
                        uint32_t(__float2int_rn(__uint_as_float(v32[c + 2]))),
                        uint32_t(__float2int_rn(__uint_as_float(v32[c + 3]))));
                __syncwarp();
                int32_t *const yi = E.y_i32;
                float *const yf = E.y_f32;
                if (vec) {
#pragma unroll 2
                    for (int k8 = 0; k8 < 8; ++k8) {
                        const int rr = k8 * 4 + (lane >> 3), c4 = (lane & 7) * 4;
                        const float xr = __shfl_sync(~0u, xs, rr);
                        const int64_t mm = mbase + rr, n = n0 + col + c4;
                        const uint4 u = *reinterpret_cast<const uint4 *>(sw + rr * kPitch + c4);
                        if (mm < E.M && n < E.N) {
                            if (yi) *reinterpret_cast<uint4 *>(yi + mm * E.N + n) = u;
                            if (yf)
                                *reinterpret_cast<float4 *>(yf + mm * E.N + n) = make_float4(
                                    dequant(int32_t(u.x), E.w_scale, xr), dequant(int32_t(u.y), E.w_scale, xr),
                                    dequant(int32_t(u.z), E.w_scale, xr), dequant(int32_t(u.w), E.w_scale, xr));
                        }
                    }
                } else {
#pragma unroll 4
                    for (int rr = 0; rr < 32; ++rr) {
                        const float xr = __shfl_sync(~0u, xs, rr);
                        const int64_t mm = mbase + rr, n = n0 + col + lane;
                        const int32_t y = int32_t(sw[rr * kPitch + lane]);
                        if (mm < E.M && n < E.N) {
                            if (yi) yi[mm * E.N + n] = y;
                            if (yf) yf[mm * E.N + n] = dequant(y, E.w_scale, xr);
                        }
                    }
                }
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_at(&tempty[a], 0);   // the leader's count
        }
    }

    // teardown: every MMA of the pair has completed before tensor memory is freed
    __syncwarp();
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp == kMmaWarp) {
        bool fin = true;
        if (lane == 0) fin = mbar_wait(done, 0, timed_out);
        fin = __shfl_sync(~0u, fin, 0);
        (void)fin;
    }
    tc_fence_before();
    cluster_sync_all();   // neither CTA frees tensor memory while the pair's MMAs may run
    tc_fence_after();
    if (threadIdx.x == 0) {   // after the last wait: every flag is set by now
        uint32_t f = 0;
        if (*timed_out) f |= TRIT_ERR_TIMEOUT;
        if (*viol_any) f |= TRIT_ERR_P1;
        if (f) atomicOr(L.err, f);
    }
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols));
}

// Row blocks of 128 of the fp16 activation copy: an even count (pair tiles).
int64_t act_blocks(const ProjDev &p) { return 2 * ((p.M + kPairM - 1) / kPairM); }

// Bytes of the blocked fp16 activation copy of one product.
int64_t act_f16_bytes(const ProjDev &p) { return act_blocks(p) * int64_t(p.B) * kBlock; }

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
    int64_t tiles = 0;
    for (int i = 0; i < n; ++i) {
        const ProjDev &p = list[i];
        const int64_t mblocks = act_blocks(p);
        CEntry &c = C.e[i];
        c.x = p.x;
        c.xh = xh[i];
        c.M = p.M;
        c.K = p.K;
        c.B = p.B;
        c.brows = kSubM;
        c.mblocks = int32_t(mblocks);
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
        E.mtiles = int32_t(mblocks / 2);
        E.ntiles = int32_t((p.N + kPairN - 1) / kPairN);
        E.w_scale = p.w_scale;
        E.pad_ = 0;
        E.tile_begin = tiles;
        tiles += int64_t(E.mtiles) * E.ntiles;
    }
    L.total_tiles = tiles;
    cudaError_t e = launch_act_f16(C, s);
    if (e != cudaSuccess) return e;
    if (tiles == 0) return cudaSuccess;
    // persistent: one pair per two SMs (at most one pair per tile)
    int64_t pairs = device_sm_count() / 2;
    pairs = pairs < tiles ? pairs : tiles;
    pairs = pairs < 1 ? 1 : pairs;
    prefill_kernel<<<dim3(unsigned(2 * pairs)), kThreads, kSmemBytes, s>>>(L);
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

namespace tc {

cudaError_t launch_act_f16(CList &C, cudaStream_t s) {
    int64_t halves = 0;
    for (int i = 0; i < C.count; ++i) {
        C.e[i].half_begin = halves;
        halves += int64_t(C.e[i].mblocks) * C.e[i].brows * 2 * C.e[i].B;
    }
    C.total = halves;
    if (halves == 0) return cudaSuccess;
    int64_t blocks = (halves + 255) / 256;
    const int64_t cap = int64_t(device_sm_count()) * 16;
    blocks = blocks < cap ? blocks : cap;
    act_f16_kernel<<<int(blocks), 256, 0, s>>>(C);
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace trit

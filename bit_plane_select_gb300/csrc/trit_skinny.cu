// Batched decode on the tensor cores: y = W x for a few activation rows
// (kSkinnyMinM <= M <= kSkinnyMaxM), the small-M case of the ternary product
// ("Tritium: One Weight Format for Ternary Inference ..." -- Introduction,
// Eq. 3; the weights in the .trit v1 plane layout, "The .trit format,
// version 1" -- 2.3).
//
// With few activation rows every weight is used M times, so the work is the
// expansion of the planes to +-1 operands, not the multiply.  The operands are
// therefore arranged the other way round from the prefill kernel: operand A
// (MMA M = 128) is a tile of 128 expanded weight rows, operand B (MMA N = nt,
// M rounded up to a multiple of 16) holds all activation rows, so no MMA work
// is spent on padding rows beyond that rounding, and the accumulator holds one
// weight row per TMEM lane and one activation row per column -- the epilogue
// stores each activation row's outputs as whole 128-byte segments without a
// transpose.
//
// Two launches per list of products:
//  1. the fp16 activation copy (trit_tc.cuh), one block of nt rows x one beat
//     per stage, nt * 128 bytes.
//  2. skinny_kernel: persistent, two CTAs per SM, tcgen05.mma.cta_group::1
//     kind::f16, M = 128, N = nt, K = 16.  Each CTA takes a contiguous range of
//     the list's tiles (128 weight rows x all K of one product), split by cost
//     (beats).  A loader warp streams the tiles' plane beats into eight raw
//     slots (16-byte cp.async, completion tracked on each slot's barrier), so
//     the producer warps issue no loads of their own (measured 4-5% faster
//     than each producer thread loading its row's beats).
//     Per stage (one beat) one thread brings the activation block with a bulk
//     copy and four producer warps (one thread per weight row) expand the
//     row's beat to fp16 +-1 in shared memory; one thread issues four MMAs per stage
//     and commits to the stage's `empty` barrier; two accumulators alternate
//     between tiles so four epilogue warps (one per TMEM lane quarter) store
//     one tile while the next is multiplied.
// Every mbarrier wait is bounded: after kWaitNs it sets TRIT_ERR_TIMEOUT and
// the roles unwind; before tensor memory is freed the CTA waits, again
// bounded, for the commit that follows its last MMA.
#include "trit_tc.cuh"

namespace trit {
namespace {

using namespace tc;

constexpr int kTileN = 128;                       // weight rows per tile (MMA M, TMEM lanes)
constexpr int kMaxNt = int(kSkinnyMaxM + 15) / 16 * 16;   // activation rows per MMA, at most
constexpr int kRaw = 8;                           // plane beats in flight (raw slots)
constexpr int kProducerWarps = 4;
constexpr int kLoaderWarp = kProducerWarps;
constexpr int kMmaWarp = kLoaderWarp + 1;
constexpr int kEpiWarp0 = kMmaWarp + 1;
constexpr int kEpiWarps = 4;                      // one per TMEM lane quarter
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr int kAStage = kTileN * kBK * 2;         // 16 KB of expanded weights
constexpr int kRawStage = kProducerWarps * 32 * 16;
constexpr int kTmemCols = 2 * kMaxNt;             // two accumulators
constexpr int kMaxStages = 8;
constexpr int kBarBytes = 512;
// dynamic shared memory of one CTA: two CTAs per SM
constexpr int kSmemBytes = 110 * 1024;
constexpr int kMaxList = TRIT_MAX_LIST_PER_LAUNCH;
static_assert(kProducerWarps * 32 == kTileN, "one producer thread per weight row");
static_assert(kTmemCols == 32 || kTmemCols == 64 || kTmemCols == 128 || kTmemCols == 256,
              "tensor memory is allocated in powers of two");
static_assert(kMaxNt <= 256 && kMaxNt % 16 == 0, "MMA N for M = 128");
static_assert((2 * kMaxStages + 2 * kRaw + 5) * 8 + 16 <= kBarBytes, "barrier area");

struct SEntry {
    const uint4 *planes;
    const uint8_t *xh;      // fp16 activation blocks: [B][nt * 128 bytes]
    const float *x_scale;
    int32_t *y_i32;
    float *y_f32;
    int64_t N;
    int64_t cost_begin;     // prefix sum of tiles * B over the list
    int32_t M, nt;          // activation rows; MMA N (M rounded up to 16)
    int32_t K, B;
    int32_t tiles;          // ceil(N / 128)
    float w_scale;
};

struct SList {
    int32_t count;
    int32_t nst;            // pipeline stages
    uint32_t *err;
    int64_t total_cost;
    int32_t stage_bytes;    // kAStage + the largest nt * 128 of the list
    int32_t pad_;
    SEntry e[kMaxList];
};
static_assert(sizeof(SList) <= 32764, "kernel parameter space");

// A tile of the list: entry e, weight rows 128*j .. 128*j+127.  Tiles are taken
// in list order; tile (e, j) starts at cost cost_begin + j*B.
struct Cursor {
    int e;
    int64_t j;
};

// The first tile whose starting cost is >= cost (e == count when none is).
__device__ __forceinline__ Cursor first_at(const SList &L, int64_t cost) {
    int a = 0, b = L.count - 1;
    while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (L.e[mid].cost_begin <= cost) a = mid;
        else b = mid - 1;
    }
    Cursor c;
    c.e = a;
    const int64_t B = L.e[a].B;
    c.j = (cost - L.e[a].cost_begin + B - 1) / B;
    if (c.j >= L.e[a].tiles) {
        c.e = a + 1;
        c.j = 0;
    }
    return c;
}

__device__ __forceinline__ bool in_range(const SList &L, const Cursor &c, int64_t end) {
    return c.e < L.count && L.e[c.e].cost_begin + c.j * L.e[c.e].B < end;
}

__device__ __forceinline__ void advance(const SList &L, Cursor &c) {
    if (++c.j == L.e[c.e].tiles) {
        ++c.e;
        c.j = 0;
    }
}

// Instruction descriptor, kind::f16: fp32 accumulator, fp16 A and B, both
// K-major, M = 128, N = nt.
__device__ __forceinline__ uint32_t idesc_128(int nt) {
    return (1u << 4) | (uint32_t(nt >> 3) << 17) | (uint32_t(kTileN >> 4) << 24);
}

__device__ __forceinline__ void mma_one(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

// Arrive on the barrier once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Arrive on the barrier once every cp.async this thread has issued has landed
// (one of the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 2) skinny_kernel(const __grid_constant__ SList L) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const int nst = L.nst;
    const int stage_bytes = L.stage_bytes;
    uint8_t *raw = smem + nst * stage_bytes;           // kRaw slots of kRawStage bytes
    uint64_t *full = reinterpret_cast<uint64_t *>(raw + kRaw * kRawStage);
    uint64_t *empty = full + kMaxStages;
    uint64_t *rfull = empty + kMaxStages;   // raw slot r holds its beat
    uint64_t *rempty = rfull + kRaw;        // raw slot r has been read
    uint64_t *tfull = rempty + kRaw;        // accumulator a holds a finished tile
    uint64_t *tempty = tfull + 2;           // accumulator a has been read
    uint64_t *done = tempty + 2;            // every MMA has completed
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    uint32_t *timed_out = tmem_slot + 1;
    uint32_t *viol_any = timed_out + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's tiles: those starting in [begin, end) of the list's cost
    const int64_t begin = L.total_cost * blockIdx.x / gridDim.x;
    const int64_t end = L.total_cost * (blockIdx.x + 1) / gridDim.x;
    const Cursor first = first_at(L, begin);

    if (threadIdx.x == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], kProducerWarps + 1);   // producer warps + the expect_tx arrival
            mbar_init(&empty[s], 1);
        }
        for (int r = 0; r < kRaw; ++r) {
            mbar_init(&rfull[r], 32);              // the loader lanes' copy completions
            mbar_init(&rempty[r], kProducerWarps);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], kEpiWarps);
        }
        mbar_init(done, 1);
        *timed_out = 0;
        *viol_any = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
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
        // thread p: weight row p of each tile; its beat comes from the raw slot
        const int p = threadIdx.x;
        uint32_t viol = 0;
        int64_t it = 0;   // stages filled
        bool stop = false;
        for (Cursor c = first; in_range(L, c, end) && !stop; advance(L, c)) {
            const SEntry &E = L.e[c.e];
            const uint32_t bbytes = uint32_t(E.nt) * 128u;
            for (int kb = 0; kb < E.B; ++kb, ++it) {
                const int s = int(it % nst);
                const uint32_t ph = uint32_t(it / nst) & 1u;
                const int r = int(it % kRaw);
                const uint32_t rph = uint32_t(it / kRaw) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, timed_out)) {
                    stop = true;
                    break;
                }
                uint8_t *a_st = smem + s * stage_bytes;
                if (p == 0) {   // the activation block of this stage
                    mbar_arrive_expect_tx(&full[s], bbytes);
                    bulk_load(a_st + kAStage, E.xh + int64_t(kb) * bbytes, bbytes, &full[s]);
                }
                if (!mbar_wait(&rfull[r], rph, timed_out)) {
                    stop = true;
                    break;
                }
                const uint4 pn = *reinterpret_cast<const uint4 *>(raw + r * kRawStage + p * 16);
                viol |= (pn.x & pn.z) | (pn.y & pn.w);
#pragma unroll
                for (int bh = 0; bh < 2; ++bh) {   // chunks 4*bh .. 4*bh+3 of row p
                    const uint32_t P = bh ? pn.y : pn.x, Q = bh ? pn.w : pn.z;
                    uint32_t w[8];
                    expand_quarter(P, Q, w);
                    *reinterpret_cast<uint4 *>(a_st + sw128_off(p, 4 * bh)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(a_st + sw128_off(p, 4 * bh + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
                    expand_quarter(P >> 8, Q >> 8, w);
                    *reinterpret_cast<uint4 *>(a_st + sw128_off(p, 4 * bh + 2)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(a_st + sw128_off(p, 4 * bh + 3)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&full[s]);
                    mbar_arrive(&rempty[r]);
                }
            }
        }
        if (viol) atomicOr(viol_any, 1u);
    } else if (warp == kLoaderWarp) {
        // lane l: weight rows l, l+32, l+64, l+96 of each tile, one beat per raw
        // slot by 16-byte cp.async (zeros past the last row); the slot's barrier
        // completes when every lane's copies have landed
        int64_t li = 0;
        bool stop = false;
        for (Cursor c = first; in_range(L, c, end) && !stop; advance(L, c)) {
            const SEntry &E = L.e[c.e];
            const uint8_t *rowp[4];
            uint32_t rbytes[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int64_t n = c.j * kTileN + lane + 32 * q;
                const bool ok = n < E.N;
                rowp[q] = reinterpret_cast<const uint8_t *>(E.planes + (ok ? n : 0) * E.B);
                rbytes[q] = ok ? 16u : 0u;
            }
            for (int kb = 0; kb < E.B; ++kb, ++li) {
                const int r = int(li % kRaw);
                const uint32_t ph = uint32_t(li / kRaw) & 1u;
                if (!mbar_wait(&rempty[r], ph ^ 1u, timed_out)) {
                    stop = true;
                    break;
                }
                uint8_t *slot = raw + r * kRawStage;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    cp_async16(slot + (lane + 32 * q) * 16, rowp[q] + int64_t(kb) * 16, rbytes[q]);
                cp_async_arrive_noinc(&rfull[r]);
            }
        }
        cp_async_wait_all();
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t base = smem_u32(smem);
            int64_t it = 0, i = 0;
            bool stop = false;
            for (Cursor c = first; in_range(L, c, end) && !stop; advance(L, c), ++i) {
                const int a = int(i & 1);
                const uint32_t use = uint32_t(i >> 1);
                if (!mbar_wait(&tempty[a], (use & 1u) ^ 1u, timed_out)) break;
                tc_fence_after();
                const SEntry &E = L.e[c.e];
                const uint32_t idesc = idesc_128(E.nt);
                const uint32_t d = tmem + uint32_t(a * kMaxNt);
                for (int kb = 0; kb < E.B; ++kb, ++it) {
                    const int s = int(it % nst);
                    const uint32_t ph = uint32_t(it / nst) & 1u;
                    if (!mbar_wait(&full[s], ph, timed_out)) {
                        stop = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = base + uint32_t(s * stage_bytes), b_addr = a_addr + kAStage;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        mma_one(d, sw128_desc(a_addr + kk * 32), sw128_desc(b_addr + kk * 32), idesc,
                                (kb > 0 || kk > 0) ? 1u : 0u);
                    mma_commit(&empty[s]);
                }
                if (!stop) mma_commit(&tfull[a]);
            }
            mma_commit(done);   // tracks every MMA issued above
        }
        __syncwarp();
    } else {
        // epilogue: warp w reads TMEM lanes 32*(w%4).. -- weight rows -- and, 16
        // activation rows at a time, stores each activation row's outputs for
        // the warp's 32 weight rows (128 contiguous bytes per store).
        const int q = warp & 3;
        int64_t i = 0;
        for (Cursor c = first; in_range(L, c, end); advance(L, c), ++i) {
            const int a = int(i & 1);
            const uint32_t use = uint32_t(i >> 1);
            const bool ok = __all_sync(~0u, mbar_wait(&tfull[a], use & 1u, timed_out));
            if (!ok) break;
            tc_fence_after();
            const SEntry &E = L.e[c.e];
            const int64_t n = c.j * kTileN + 32 * q + lane;
            const bool live = n < E.N;
            int32_t *const yi = E.y_i32;
            float *const yf = E.y_f32;
#pragma unroll 1
            for (int t0 = 0; t0 < E.nt; t0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem + (uint32_t(32 * q) << 16) + uint32_t(a * kMaxNt + t0), v);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int t = t0 + k;
                    if (t < E.M && live) {
                        const int32_t y = __float2int_rn(__uint_as_float(v[k]));
                        if (yi) yi[int64_t(t) * E.N + n] = y;
                        if (yf) yf[int64_t(t) * E.N + n] = dequant(y, E.w_scale, E.x_scale[t]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[a]);
        }
    }

    // teardown: every MMA has completed before tensor memory is freed
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) {
        bool fin = true;
        if (lane == 0) fin = mbar_wait(done, 0, timed_out);
        fin = __shfl_sync(~0u, fin, 0);
        (void)fin;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {   // after the last wait: every flag is set by now
        uint32_t f = 0;
        if (*timed_out) f |= TRIT_ERR_TIMEOUT;
        if (*viol_any) f |= TRIT_ERR_P1;
        if (f) atomicOr(L.err, f);
    }
    if (warp == kMmaWarp)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

int nt_of(int64_t M) { return int((M + 15) / 16 * 16); }

// Bytes of the fp16 activation copy of one product: one block of nt rows per beat.
int64_t act_bytes(const ProjDev &p) { return int64_t(nt_of(p.M)) * 128 * p.B; }

cudaError_t set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(skinny_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(skinny_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

// Convert and multiply the products list[0..n) with their fp16 activation
// copies at xh[i] (each act_bytes long, 16-byte aligned).
cudaError_t launch_two(const ProjDev *list, int n, uint8_t *const *xh, uint32_t *err, cudaStream_t s) {
    static thread_local CList C;
    static thread_local SList L;
    C.count = n;
    C.pad_ = 0;
    L.count = n;
    L.err = err;
    L.pad_ = 0;
    int64_t cost = 0, tiles = 0;
    int maxnt = 16;
    for (int i = 0; i < n; ++i) {
        const ProjDev &p = list[i];
        const int nt = nt_of(p.M);
        CEntry &c = C.e[i];
        c.x = p.x;
        c.xh = xh[i];
        c.M = p.M;
        c.K = p.K;
        c.B = p.B;
        c.brows = nt;
        c.mblocks = 1;
        SEntry &E = L.e[i];
        E.planes = p.planes;
        E.xh = xh[i];
        E.x_scale = p.x_scale;
        E.y_i32 = p.y_i32;
        E.y_f32 = p.y_f32;
        E.N = p.N;
        E.cost_begin = cost;
        E.M = int32_t(p.M);
        E.nt = nt;
        E.K = p.K;
        E.B = p.B;
        E.tiles = int32_t((p.N + kTileN - 1) / kTileN);
        E.w_scale = p.w_scale;
        cost += int64_t(E.tiles) * p.B;
        tiles += E.tiles;
        maxnt = nt > maxnt ? nt : maxnt;
    }
    L.total_cost = cost;
    L.stage_bytes = kAStage + maxnt * 128;
    const int room = kSmemBytes - 1024 - kRaw * kRawStage - kBarBytes;
    L.nst = room / L.stage_bytes < kMaxStages ? room / L.stage_bytes : kMaxStages;
    cudaError_t e = launch_act_f16(C, s);
    if (e != cudaSuccess) return e;
    if (tiles == 0) return cudaSuccess;
    // persistent: two CTAs per SM, at most one per tile
    int64_t ctas = 2 * int64_t(device_sm_count());
    ctas = ctas < tiles ? ctas : tiles;
    skinny_kernel<<<unsigned(ctas), kThreads, kSmemBytes, s>>>(L);
    return cudaGetLastError();
}

}  // namespace

bool skinny_supported(const ProjDev &p) {
    return p.M >= kSkinnyMinM && p.M <= kSkinnyMaxM && p.K < 131072;
}

int64_t skinny_scratch_bytes(const ProjDev &p) { return act_bytes(p); }

cudaError_t launch_skinny_into(const ProjDev &p, uint8_t *xh, uint32_t *err, cudaStream_t s) {
    cudaError_t e = set_attributes();
    if (e != cudaSuccess) return e;
    uint8_t *const one[1] = {xh};
    return launch_two(&p, 1, one, err, s);
}

// The fp16 activation copies are allocated stream-ordered (cudaMallocAsync on
// `s`) and freed after the launches, in groups of at most kScratchGroup bytes.
cudaError_t launch_skinny_many(const ProjDev *list, int count, uint32_t *err, cudaStream_t s) {
    constexpr int64_t kScratchGroup = int64_t(1) << 30;
    cudaError_t ae = set_attributes();
    if (ae != cudaSuccess) return ae;
    static thread_local uint8_t *xh[kMaxList];
    int base = 0;
    while (base < count) {
        int n = 0;
        int64_t bytes = 0;
        while (base + n < count && n < kMaxList) {
            const int64_t b = (act_bytes(list[base + n]) + 255) & ~int64_t(255);
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
            off += (act_bytes(list[base + i]) + 255) & ~int64_t(255);
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

"""trit_gemm_noalloc, the entry point that allocates nothing, against
trit_gemm and against the CPU oracle on the same inputs: two calls in a row on
one stream (the second reusing the fixed scratch the first one wrote) must
each give trit_gemm's bits, and the oracle's on sampled rows.  The device's
memory pool must not grow during the calls (trit_gemm on the same product
does grow it: the control).  Also: a product whose activation copy does not
fit the fixed buffer is refused before anything is enqueued, and a
both-bits-set beat is flagged the same way.  The file sorts last so that it
also runs after everything else."""
import ctypes

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def t():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_plane_select_gb300 import build
    build.build()
    import bit_plane_select_gb300 as t
    torch.cuda.set_device(0)
    return t


def scratch_bytes(M, K):
    """Bytes of the fp16 activation copy the tensor-core paths need: for
    M <= 128 one block of M rows (rounded up to 16) x 64 columns per beat; above,
    16 KB blocks of 128 rows x 64 columns, row blocks in pairs (256-row pair
    tiles)."""
    if M < 13 or K >= 131072:
        return 0
    if M <= 128:
        return 128 * ((M + 15) // 16 * 16) * ((K + 63) // 64)
    return 32768 * ((M + 255) // 256) * ((K + 63) // 64)


def make_product(t, M, N, K, seed):
    rng = synth.rng_for(900, M, N, K, seed)
    w = synth.ternary(rng, N, K, synth.P_ZERO)
    ws = float(synth.w_scale(w))
    planes, err = t.trit_pack(torch.from_numpy(w).cuda(), ws)
    kp = ((K + 63) // 64) * 64
    x = np.zeros((M, kp), np.int8)
    x[:, :K] = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    xs = rng.uniform(0.05, 8.0, size=M).astype(np.float32)
    return dict(planes=planes, ws=ws, x=torch.from_numpy(x).cuda(),
                xs=torch.from_numpy(xs).cuda(), M=M, N=N, K=K, w=w, xh=x, xsh=xs)


def oracle_rows(N, seed):
    """About 24 output rows to compare with the oracle: the first, the last and
    a seeded sample between them."""
    rng = np.random.default_rng(seed)
    rows = set(int(r) for r in rng.choice(N, size=min(N, 22), replace=False))
    return np.array(sorted(rows | {0, N - 1}), dtype=np.int64)


def matches_oracle(P, got, seed):
    torch.cuda.synchronize()
    rows = oracle_rows(P["N"], seed)
    ry, rf, rerr = oracle.gemm(oracle.pack(P["w"]), P["ws"], P["xh"], P["xsh"], P["K"], rows=rows)
    assert not rerr.any()
    y32, yf = got[0].cpu().numpy(), got[1].cpu().numpy()
    np.testing.assert_array_equal(y32[:, rows], ry)
    np.testing.assert_array_equal(yf[:, rows].view(np.uint32), rf.view(np.uint32))


def outputs(P):
    dev = P["planes"].device
    y32 = torch.full((P["M"], P["N"]), 0x5A5A5A5A, dtype=torch.int32, device=dev)
    yf = torch.full((P["M"], P["N"]), float("nan"), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    return y32, yf, err


def via_noalloc(t, P):
    y32, yf, err = outputs(P)
    t.trit_gemm_noalloc(P["planes"], P["ws"], P["x"], P["xs"], P["K"], y32, yf, err)
    return y32, yf, err


def via_gemm(t, P):
    y32, yf, err = outputs(P)
    t.trit_gemm(P["planes"], P["ws"], P["x"], P["xs"], P["K"], y_i32=y32, y_f32=yf, err_flag=err)
    return y32, yf, err


def same(a, b):
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u.cpu().view(torch.int32), v.cpu().view(torch.int32))


# (first product, second product): the second call runs right after the first
# on the same stream and reuses the buffer the first one filled.
PAIRS = [
    ((300, 200, 1000), (40, 129, 65)),          # tensor path, ragged tiles; smaller second call
    ((2048, 256, 6912), (517, 300, 2560)),      # a prefill-sized product, 27 MiB of scratch
    ((2048, 136, 8192), (2048, 136, 8192)),     # exactly the whole 32 MiB buffer, twice
    ((5, 300, 2560), (1, 700, 6913)),           # integer paths (no scratch)
    ((40, 64, 140000), (13, 33, 64)),           # K past the tensor path, then the smallest M on it
    ((128, 300, 131071), (129, 300, 2560)),     # largest small-M copy (32 MiB), then a pair-tile one
]


@pytest.mark.parametrize("first,second", PAIRS)
def test_two_calls_in_a_row_match_trit_gemm(t, first, second):
    A = make_product(t, *first, seed=1)
    B = make_product(t, *second, seed=2)
    assert scratch_bytes(first[0], first[2]) <= t.NOALLOC_SCRATCH_BYTES
    ra = via_noalloc(t, A)
    rb = via_noalloc(t, B)
    ea = via_gemm(t, A)
    eb = via_gemm(t, B)
    same(ra, ea)
    same(rb, eb)
    assert int(ra[2].item()) == 0 and int(rb[2].item()) == 0
    matches_oracle(A, ra, 11)
    matches_oracle(B, rb, 12)


# ---- the device's default memory pool (driver API, read through libcuda) ----
# cudaMallocAsync, the allocator trit_gemm's tensor-core paths use, draws from
# the device's current memory pool -- the default one unless someone replaced
# it; torch's caching allocator does not use it.  The pool's high-water mark of
# memory in use is reset to 0 before the calls and read after them.
CU_MEMPOOL_ATTR_USED_MEM_HIGH = 8


def _driver():
    try:
        return ctypes.CDLL("libcuda.so.1")
    except OSError:
        pytest.skip("libcuda.so.1 not found")


def pool_used_high(reset=False):
    cu = _driver()
    dev = ctypes.c_int(0)
    assert cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
    pool = ctypes.c_void_p(0)
    assert cu.cuDeviceGetDefaultMemPool(ctypes.byref(pool), dev) == 0
    v = ctypes.c_uint64(0)
    if reset:
        assert cu.cuMemPoolSetAttribute(pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(v)) == 0
    assert cu.cuMemPoolGetAttribute(pool, CU_MEMPOOL_ATTR_USED_MEM_HIGH, ctypes.byref(v)) == 0
    return int(v.value)


@pytest.mark.parametrize("first,second", [PAIRS[0], PAIRS[1], PAIRS[5]])
def test_no_pool_growth(t, first, second):
    """Two tensor-core products through trit_gemm_noalloc leave the pool's
    high-water mark at zero; the same two through trit_gemm raise it."""
    A = make_product(t, *first, seed=7)
    B = make_product(t, *second, seed=8)
    torch.cuda.synchronize()
    assert pool_used_high(reset=True) == 0
    via_noalloc(t, A)
    via_noalloc(t, B)
    torch.cuda.synchronize()
    assert pool_used_high() == 0, "trit_gemm_noalloc drew memory from the device pool"
    via_gemm(t, A)
    via_gemm(t, B)
    torch.cuda.synchronize()
    assert pool_used_high() > 0, "control: trit_gemm's tensor-core path allocates on the stream"


def test_limit_counts_row_blocks_in_pairs(t):
    """M = 1920 (15 blocks of 128 rows, padded to 16) with K = 8192 (128 beats)
    needs exactly 32 MiB and runs; K = 8193 (129 beats) does not."""
    M, N = 1920, 8
    assert scratch_bytes(M, 8192) == t.NOALLOC_SCRATCH_BYTES
    assert scratch_bytes(M, 8193) > t.NOALLOC_SCRATCH_BYTES
    P = make_product(t, M, N, 8192, seed=5)
    same(via_noalloc(t, P), via_gemm(t, P))
    Q = make_product(t, M, N, 8193, seed=6)
    y32, yf, err = outputs(Q)
    with pytest.raises(t.TritError) as info:
        t.trit_gemm_noalloc(Q["planes"], Q["ws"], Q["x"], Q["xs"], Q["K"], y32, yf, err)
    assert info.value.status == 8


def test_one_output_only(t):
    P = make_product(t, 100, 96, 777, seed=3)
    y32, _, err = outputs(P)
    t.trit_gemm_noalloc(P["planes"], P["ws"], P["x"], P["xs"], P["K"], y32, None, err)
    ref = via_gemm(t, P)
    torch.cuda.synchronize()
    assert torch.equal(y32.cpu(), ref[0].cpu())


def test_oversized_product_is_refused(t):
    M, N, K = 2048, 8, 8193          # 16 * 129 blocks: 33 MiB > 32 MiB
    assert scratch_bytes(M, K) > t.NOALLOC_SCRATCH_BYTES
    P = make_product(t, M, N, K, seed=4)
    y32, yf, err = outputs(P)
    torch.cuda.synchronize()
    with pytest.raises(t.TritError) as info:
        t.trit_gemm_noalloc(P["planes"], P["ws"], P["x"], P["xs"], K, y32, yf, err)
    assert info.value.status == 8
    torch.cuda.synchronize()
    assert bool((y32 == 0x5A5A5A5A).all()) and bool(torch.isnan(yf).all())
    assert int(err.item()) == 0
    # the same product split in two halves of M fits
    for lo in (0, M // 2):
        h = dict(P, x=P["x"][lo:lo + M // 2].contiguous(), xs=P["xs"][lo:lo + M // 2].contiguous(),
                 M=M // 2)
        same(via_noalloc(t, h), via_gemm(t, h))


def test_both_set_beat_flagged_like_trit_gemm(t):
    P = make_product(t, 64, 50, 300, seed=5)
    pl = P["planes"].cpu().numpy().copy()
    pl[7, 2, 8:16] = pl[7, 2, 0:8]           # beat 2 of row 7: neg := pos
    pl[7, 2, 0] |= 1
    pl[7, 2, 8] |= 1
    P["planes"] = torch.from_numpy(pl).cuda()
    ra = via_noalloc(t, P)
    rb = via_gemm(t, P)
    torch.cuda.synchronize()
    assert int(ra[2].item()) & 1 and int(ra[2].item()) == int(rb[2].item())
    keep = [r for r in range(P["N"]) if r != 7]
    assert torch.equal(ra[0][:, keep].cpu(), rb[0][:, keep].cpu())
    assert torch.equal(ra[1][:, keep].cpu().view(torch.int32), rb[1][:, keep].cpu().view(torch.int32))

"""GPU parity: every entry point of the C ABI against the CPU oracle, element
by element, on seeded inputs that span several tiles and ragged tails, plus
the edge cases (one row, one column, K % 64 != 0, the largest K, -128
activations, both-bits-set beats, dirty padding, non-finite activations).

Integer results must be bit-exact; fp32 outputs within 1e-6 relative (they
are in fact expected bit-identical, checked separately)."""
import numpy as np
import pytest

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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(x):
    torch.cuda.synchronize()
    return x.cpu().numpy()


def assert_f32_close(got, ref, tol=1e-6):
    """Relative error <= tol; identical values (infinities included) match."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    with np.errstate(invalid="ignore"):
        rel = np.where(got == ref, 0.0, np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30))
    assert not np.isnan(rel).any()
    assert float(rel.max(initial=0.0)) <= tol


def padded_x(rng, M, K, fill=0):
    kp = ((K + 63) // 64) * 64
    x = np.full((M, kp), fill, np.int8)
    x[:, :K] = rng.integers(-128, 128, size=(M, K)).astype(np.int8)
    return x


# ---- layout ---------------------------------------------------------------

LAYOUT_SHAPES = [(1, 1), (3, 63), (16, 64), (17, 65), (40, 127), (33, 2560), (7, 6912), (641, 200)]


@pytest.mark.parametrize("N,K", LAYOUT_SHAPES)
def test_pack_unpack_verify(t, orc, N, K):
    rng = synth.rng_for(100, N, K)
    w = synth.ternary(rng, N, K, synth.P_ZERO)
    planes, err = t.trit_pack(dev(w), 0.5)
    np.testing.assert_array_equal(host(planes), orc.pack(w))
    back, err = t.trit_unpack(planes, K, err_flag=err)
    np.testing.assert_array_equal(host(back), w)
    err, first = t.trit_verify(planes, K, err_flag=err)
    assert int(host(err)[0]) == 0 and int(host(first)[0]) == -1


def test_pack_scale_out_and_guard(t):
    N, K = 9, 130
    w = synth.ternary(synth.rng_for(101), N, K, 0.4)
    B = (K + 63) // 64
    buf = torch.full((N * B * 16 + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    planes = buf[:N * B * 16].view(N, B, 16)
    scale = torch.zeros(2, dtype=torch.float32, device="cuda")
    t.trit_pack(dev(w), 0.375, planes=planes, scale_out=scale[:1])
    tail = host(buf)[N * B * 16:]
    assert (tail == 0xA5).all()
    assert host(scale).tolist() == [0.375, 0.0]


def test_pack_flags_non_ternary(t):
    w = np.zeros((5, 100), np.int8)
    w[3, 77] = 2
    w[1, 5] = -128
    planes, err = t.trit_pack(dev(w), 1.0)
    assert int(host(err)[0]) == t.ERR_NOT_TERNARY
    w_ok = np.zeros((5, 100), np.int8)
    planes, err = t.trit_pack(dev(w_ok), 1.0)
    assert int(host(err)[0]) == 0


@pytest.mark.parametrize("K", [64, 100, 130, 191])
def test_verify_matches_oracle_on_corruption(t, orc, K):
    rng = synth.rng_for(102, K)
    N = 50
    p = orc.pack(synth.ternary(rng, N, K, 0.4))
    B = p.shape[1]
    cases = []
    for trial in range(6):
        q = p.copy()
        r = int(rng.integers(0, N))
        b = int(rng.integers(0, B))
        k = int(rng.integers(0, 64))
        kind = trial % 3
        if kind == 0:      # both planes at one position
            q[r, b, k // 8] |= 1 << (k % 8)
            q[r, b, 8 + k // 8] |= 1 << (k % 8)
        elif kind == 1 and K % 64:   # a padding bit
            kk = int(rng.integers(K % 64, 64))
            q[r, B - 1, 8 * int(rng.integers(0, 2)) + kk // 8] |= 1 << (kk % 8)
        cases.append(q)
    cases.append(p.copy())
    for q in cases:
        kinds, first = orc.verify(q, K)
        err, fb = t.trit_verify(dev(q), K)
        assert int(host(err)[0]) == kinds
        assert int(host(fb)[0]) == first
        if kinds & orc.P1:
            _, uerr = t.trit_unpack(dev(q), K)
            assert int(host(uerr)[0]) == t.ERR_P1


# ---- quantiser ------------------------------------------------------------

def quant_cases(rng, K):
    x = rng.standard_normal((8, K)).astype(np.float32)
    x[1] = 0.0                                          # zero row
    x[2] = (rng.integers(-127, 128, K) * 2.0 ** -140).astype(np.float32)   # denormal row
    x[3] = np.round(rng.standard_normal(K) * 40) / 2    # many exact ties
    x[3, 0] = 127.0
    x[4] *= np.float32(1e37)                            # large magnitudes
    x[5, K // 2] = np.nan
    x[6, K - 1] = -np.inf
    x[7] = -x[7]
    return x


@pytest.mark.parametrize("K", [1, 63, 64, 65, 2560, 6912])
def test_quant_matches_oracle(t, orc, K):
    rng = synth.rng_for(103, K)
    x = quant_cases(rng, K)
    q_ref, s_ref, e_ref = orc.quant(x)
    kp = q_ref.shape[1]
    q = torch.full((8, kp), 99, dtype=torch.int8, device="cuda")   # tail must be overwritten
    q, s, err = t.trit_quant_act(dev(x), x_i8=q)
    np.testing.assert_array_equal(host(q), q_ref)
    np.testing.assert_array_equal(host(s), s_ref)
    want_flag = t.ERR_NONFINITE if e_ref.any() else 0
    assert int(host(err)[0]) == want_flag


def test_quant_many_matches_single(t, orc):
    rng = synth.rng_for(104)
    xs = [rng.standard_normal((m, k)).astype(np.float32) for m, k in [(1, 2560), (3, 6912), (2, 65)]]
    outs = [(dev(x), torch.empty((x.shape[0], ((x.shape[1] + 63) // 64) * 64), dtype=torch.int8,
                                 device="cuda"), torch.empty(x.shape[0], dtype=torch.float32,
                                                             device="cuda")) for x in xs]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t.trit_quant_act_many(t.ActList(outs), err)
    for x, (_, q, s) in zip(xs, outs):
        q_ref, s_ref, _ = orc.quant(x)
        np.testing.assert_array_equal(host(q), q_ref)
        np.testing.assert_array_equal(host(s), s_ref)


# ---- products -------------------------------------------------------------

GEMM_CASES = [
    (1, 1, 1), (1, 3, 63), (1, 4, 64), (1, 5, 65), (1, 33, 200), (1, 257, 2560), (1, 1000, 6912),
    (1, 127, 1000), (2, 37, 130), (3, 64, 2560), (4, 33, 6912), (5, 100, 65), (7, 17, 640),
    (8, 260, 2560), (9, 45, 300), (12, 77, 1000), (13, 70, 2560), (16, 70, 2560), (17, 31, 191), (33, 9, 6912),
    # M > 1 with many 32-row groups per CTA (warp shares cut groups at step
    # boundaries), the 8 + 2 and 8 + 4 row chunkings, ragged N, and rows long
    # enough to be cut into column segments at 8 and at 2 rows
    (2, 6912, 2560), (3, 2560, 6912), (6, 2048, 2560), (10, 1000, 6912), (11, 2049, 2560),
    (12, 640, 2560), (9, 50, 20000), (4, 96, 18500),
]


def run_case(t, orc, M, N, K, seed, p0=synth.P_ZERO, x=None):
    rng = synth.rng_for(105, M, N, K, seed)
    w = synth.ternary(rng, N, K, p0)
    if x is None:
        x = padded_x(rng, M, K, fill=0)
        x[:, K:] = rng.integers(-128, 128, size=(M, x.shape[1] - K))  # garbage past K is ignored
    xs = (rng.random(M) * 3 + 0.01).astype(np.float32)
    ws = float(synth.w_scale(w))
    planes, _ = t.trit_pack(dev(w), ws)
    y, f, err = t.trit_gemm(planes, ws, dev(x), dev(xs), K)
    ry, rf, rerr = orc.gemm(orc.pack(w), ws, x, xs, K)
    assert not rerr.any()
    return host(y), host(f), int(host(err)[0]), ry, rf


@pytest.mark.parametrize("M,N,K", GEMM_CASES)
def test_gemm_matches_oracle(t, orc, M, N, K):
    y, f, err, ry, rf = run_case(t, orc, M, N, K, 0)
    assert err == 0
    np.testing.assert_array_equal(y, ry)
    assert_f32_close(f, rf)


def test_fp32_outputs_bit_identical(t, orc):
    for M, N, K in [(1, 300, 2560), (4, 129, 6912), (9, 40, 100)]:
        y, f, err, ry, rf = run_case(t, orc, M, N, K, 1)
        np.testing.assert_array_equal(f.view(np.uint32), rf.view(np.uint32))


def test_gemv_entry_point(t, orc):
    rng = synth.rng_for(106)
    N, K = 515, 2560
    w = synth.ternary(rng, N, K, 0.45)
    x = padded_x(rng, 1, K)
    xs = np.array([1.5], np.float32)
    planes, _ = t.trit_pack(dev(w), 2.0)
    y, f, err = t.trit_gemv(planes, 2.0, dev(x), float(xs[0]), K)
    ry, rf, _ = orc.gemm(orc.pack(w), 2.0, x, xs, K)
    np.testing.assert_array_equal(host(y), ry[0])
    assert_f32_close(host(f), rf[0])


@pytest.mark.parametrize("N,K,xs", [(515, 2560, 1.5), (77, 6912, 0.0), (9, 73793, 3.25),
                                    (33, 100, 1e-30)])
def test_gemv_scale_by_value(t, orc, N, K, xs):
    """trit_gemv takes the activation scale by value: the same bits as the
    oracle and as trit_gemm (M = 1) with the scale in device memory -- also for
    rows longer than one column segment (K > 73,728), whose fp32 outputs come
    from the separate dequantisation pass, and for a zero scale."""
    rng = synth.rng_for(107, K)
    w = synth.ternary(rng, N, K, 0.42)
    x = padded_x(rng, 1, K)
    xsa = np.array([xs], np.float32)
    planes, _ = t.trit_pack(dev(w), 0.75)
    y, f, err = t.trit_gemv(planes, 0.75, dev(x), xs, K)
    y2, f2, err2 = t.trit_gemm(planes, 0.75, dev(x), dev(xsa), K)
    ry, rf, _ = orc.gemm(orc.pack(w), 0.75, x, xsa, K)
    assert int(host(err)[0]) == 0 and int(host(err2)[0]) == 0
    np.testing.assert_array_equal(host(y), ry[0])
    np.testing.assert_array_equal(host(f).view(np.uint32), rf[0].view(np.uint32))
    np.testing.assert_array_equal(host(y2).reshape(-1), host(y))
    np.testing.assert_array_equal(host(f2).reshape(-1).view(np.uint32), host(f).view(np.uint32))


@pytest.mark.parametrize("K", [64, 6912, 6913])
def test_extremes(t, orc, K):
    """Rows of all +1 / all -1 / alternating against -128 and 127 activations:
    -128 must be widened before it is negated ("Tritium ..." -- The hardware
    core), and the 6912-column row of -1 against -128 gives +884,736."""
    w = np.stack([np.full(K, 1), np.full(K, -1), np.resize([1, -1, 0], K),
                  np.zeros(K)]).astype(np.int8)
    x = np.zeros((3, ((K + 63) // 64) * 64), np.int8)
    x[0, :K] = -128
    x[1, :K] = 127
    x[2, :K] = np.resize([-128, 127], K)
    xs = np.ones(3, np.float32)
    planes, _ = t.trit_pack(dev(w), 1.0)
    for M in (1, 3):
        y, f, err = t.trit_gemm(planes, 1.0, dev(x[:M]), dev(xs[:M]), K)
        ry, rf, _ = orc.gemm(orc.pack(w), 1.0, x[:M], xs[:M], K)
        np.testing.assert_array_equal(host(y), ry)
    if K == 6912:
        assert int(ry[0, 1]) == 884736


def test_largest_k(t, orc):
    """K = 2^24 - 1: |y| reaches 128*K = 2,147,483,520, just inside int32, and the
    per-lane accumulators are folded many times within one row."""
    K = (1 << 24) - 1
    w = np.stack([np.full(K, -1, np.int8), synth.ternary(synth.rng_for(107), 1, K, 0.4)[0]])
    x = np.zeros((1, ((K + 63) // 64) * 64), np.int8)
    x[0, :K] = -128
    planes, _ = t.trit_pack(dev(w), 1.0)
    y, f, err = t.trit_gemm(planes, 1.0, dev(x), dev(np.ones(1, np.float32)), K)
    ry, rf, _ = orc.gemm(orc.pack(w), 1.0, x, np.ones(1, np.float32), K)
    assert int(ry[0, 0]) == 128 * K
    np.testing.assert_array_equal(host(y), ry)


def test_long_rows_fold_accumulators(t, orc):
    K = 2_100_001      # ceil(B/8) > 4096 steps per row: exercises the mid-row fold
    rng = synth.rng_for(108)
    w = synth.ternary(rng, 5, K, 0.3)
    x = padded_x(rng, 1, K)
    planes, _ = t.trit_pack(dev(w), 1.0)
    y, f, err = t.trit_gemm(planes, 1.0, dev(x), dev(np.ones(1, np.float32)), K)
    ry, _, _ = orc.gemm(orc.pack(w), 1.0, x, np.ones(1, np.float32), K)
    np.testing.assert_array_equal(host(y), ry)


def test_outputs_optional_and_guarded(t, orc):
    rng = synth.rng_for(109)
    M, N, K = 3, 77, 300
    w = synth.ternary(rng, N, K, 0.4)
    x = padded_x(rng, M, K)
    xs = np.ones(M, np.float32)
    planes, _ = t.trit_pack(dev(w), 1.0)
    ry, rf, _ = orc.gemm(orc.pack(w), 1.0, x, xs, K)
    g = 1000
    yb = torch.full((M * N + g,), -7, dtype=torch.int32, device="cuda")
    fb = torch.full((M * N + g,), -7.0, dtype=torch.float32, device="cuda")
    t.trit_gemm(planes, 1.0, dev(x), dev(xs), K, y_i32=yb[:M * N].view(M, N), want=())
    t.trit_gemm(planes, 1.0, dev(x), dev(xs), K, y_f32=fb[:M * N].view(M, N), want=())
    yh, fh = host(yb), host(fb)
    np.testing.assert_array_equal(yh[:M * N].reshape(M, N), ry)
    assert_f32_close(fh[:M * N].reshape(M, N), rf)
    assert (yh[M * N:] == -7).all() and (fh[M * N:] == -7.0).all()


def test_both_set_beats_flagged_other_rows_exact(t, orc):
    rng = synth.rng_for(110)
    for M in (1, 4):
        N, K = 300, 2560
        w = synth.ternary(rng, N, K, synth.P_ZERO)
        p = orc.pack(w)
        bad_rows = [0, 17, 299]
        for r in bad_rows:
            b, k = int(rng.integers(0, p.shape[1])), int(rng.integers(0, 64))
            p[r, b, k // 8] |= 1 << (k % 8)
            p[r, b, 8 + k // 8] |= 1 << (k % 8)
        x = padded_x(rng, M, K)
        xs = np.ones(M, np.float32)
        y, f, err = t.trit_gemm(dev(p), 1.0, dev(x), dev(xs), K)
        ry, rf, rerr = orc.gemm(p, 1.0, x, xs, K)
        assert int(host(err)[0]) == t.ERR_P1
        assert sorted(np.nonzero(rerr)[0].tolist()) == bad_rows
        keep = rerr == 0
        np.testing.assert_array_equal(host(y)[:, keep], ry[:, keep])


def test_dirty_padding_does_not_change_products(t, orc):
    """Padding columns do not exist: a set padding bit (a P2 violation, caught by
    trit_verify) contributes nothing to y and raises no P1 flag."""
    rng = synth.rng_for(111)
    N, K = 20, 100
    w = synth.ternary(rng, N, K, 0.4)
    p = orc.pack(w)
    p[:, -1, 7] |= 0x80            # pos bit 63 of every last beat (column 127 >= 100)
    x = padded_x(rng, 2, K)
    x[:, K:] = 5
    xs = np.ones(2, np.float32)
    y, f, err = t.trit_gemm(dev(p), 1.0, dev(x), dev(xs), K)
    ry, rf, rerr = orc.gemm(p, 1.0, x, xs, K)
    assert not rerr.any() and int(host(err)[0]) == 0
    np.testing.assert_array_equal(host(y), ry)
    verr, _ = t.trit_verify(dev(p), K)
    assert int(host(verr)[0]) == t.ERR_P2


def test_gemm_many_mixed_list(t, orc):
    rng = synth.rng_for(112)
    shapes = [(1, 2560, 2560), (1, 640, 2560), (3, 100, 6912), (1, 7, 65), (8, 333, 2560),
              (2, 1, 1), (1, 6912, 2560), (5, 40, 640)]
    entries, refs = [], []
    for M, N, K in shapes:
        w = synth.ternary(rng, N, K, float(rng.uniform(0.385, 0.508)))
        x = padded_x(rng, M, K)
        xs = (rng.random(M) + 0.5).astype(np.float32)
        ws = float(synth.w_scale(w))
        planes, _ = t.trit_pack(dev(w), ws)
        y = torch.empty((M, N), dtype=torch.int32, device="cuda")
        f = torch.empty((M, N), dtype=torch.float32, device="cuda")
        entries.append((planes, ws, dev(x), dev(xs), K, y, f))
        refs.append(orc.gemm(orc.pack(w), ws, x, xs, K))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t.trit_gemm_many(t.ProjList(entries), err)
    assert int(host(err)[0]) == 0
    for (_, _, _, _, _, y, f), (ry, rf, _) in zip(entries, refs):
        np.testing.assert_array_equal(host(y), ry)
        assert_f32_close(host(f), rf)


# ---- small lists: every warp one group, planes copied to shared memory -------

def _m1_list(t, orc, rng, shapes, ready, fused):
    """M = 1 products of the given (N, K) shapes in one list call, against the
    oracle; fused: fp32 rows through trit_quant_gemv_many, else int8 rows
    through trit_gemm_many."""
    entries, refs = [], []
    for N, K in shapes:
        w = synth.ternary(rng, N, K, float(rng.uniform(0.385, 0.508)))
        ws = float(synth.w_scale(w))
        planes, _ = t.trit_pack(dev(w), ws)
        y = torch.empty(N, dtype=torch.int32, device="cuda")
        f = torch.empty(N, dtype=torch.float32, device="cuda")
        if fused:
            x = rng.standard_normal(K).astype(np.float32)
            q = torch.full((((K + 63) // 64) * 64,), 55, dtype=torch.int8, device="cuda")
            s = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
            entries.append((planes, ws, dev(x), q, s, y, f))
            q_ref, s_ref, _ = orc.quant(x[None, :])
            ry, rf, _ = orc.gemm(orc.pack(w), ws, q_ref, s_ref, K)
            refs.append((q_ref[0], s_ref, ry[0], rf[0]))
        else:
            x = padded_x(rng, 1, K)
            xs = (rng.random(1) + 0.5).astype(np.float32)
            entries.append((planes, ws, dev(x), dev(xs), K, y, f))
            ry, rf, _ = orc.gemm(orc.pack(w), ws, x, xs, K)
            refs.append((None, None, ry[0], rf[0]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if ready:
        torch.cuda.synchronize()
    if fused:
        t.trit_quant_gemv_many(t.QProjList(entries, planes_ready=ready), err)
    else:
        t.trit_gemm_many(t.ProjList(entries, planes_ready=ready), err)
    assert int(host(err)[0]) == 0
    for e, (q_ref, s_ref, ry, rf) in zip(entries, refs):
        y, f = e[5], e[6]
        if fused:
            np.testing.assert_array_equal(host(e[3]), q_ref)
            np.testing.assert_array_equal(host(e[4]), s_ref)
        np.testing.assert_array_equal(host(y), ry)
        np.testing.assert_array_equal(host(f).view(np.uint32), rf.view(np.uint32))


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("ready", [False, True])
def test_small_list_entry_boundaries(t, orc, ready, fused):
    """Entries of 1-3 groups, so that CTAs of eight warps hold the ends of
    several entries (staging each in turn), ragged rows and tails."""
    rng = synth.rng_for(130, int(ready), int(fused))
    shapes = [(3, 2560), (9, 2560), (17, 2560), (1, 2560), (8, 2560), (23, 2560), (5, 2560),
              (64, 2560), (2, 2560)]
    _m1_list(t, orc, rng, shapes, ready, fused)


@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("K", [1, 100, 6912, 13312, 13376])
def test_small_list_row_lengths(t, orc, K, fused):
    """Rows from one column to past the shared-memory limit of the
    pre-loading launch (13,312 columns take it, 13,376 the streaming kernel)."""
    rng = synth.rng_for(131, K, int(fused))
    _m1_list(t, orc, rng, [(77, K), (1, K), (130, K)], True, fused)


@pytest.mark.parametrize("N", [19456, 19464])
def test_small_list_one_wave_boundary(t, orc, N):
    """2,432 groups of 2,560 columns fill two CTAs on each of 152 SMs (the
    pre-loading launch); 2,433 do not and take the streaming kernel."""
    rng = synth.rng_for(132, N)
    _m1_list(t, orc, rng, [(N, 2560)], True, True)


def test_error_status_raises(t):
    x = torch.zeros((1, 64), dtype=torch.int8, device="cuda")
    planes = torch.zeros((4, 1, 16), dtype=torch.uint8, device="cuda")
    xs = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(t.TritError) as e:
        t.trit_gemm(planes, float("nan"), x, xs, 64)
    assert e.value.status == 4
    with pytest.raises(t.TritError) as e:
        t.trit_gemm(planes, 1.0, x, xs, 1 << 24)
    assert e.value.status == 2


# ---- fused quantise-and-multiply --------------------------------------------

FUSED_K = [1, 65, 200, 2560, 6912, 6913, 40000, 73728]


@pytest.mark.parametrize("ready", [False, True])
@pytest.mark.parametrize("K", FUSED_K)
def test_quant_gemv_many_matches_oracle(t, orc, K, ready):
    """One launch quantises each fp32 row and multiplies it: codes, scale and
    products equal the oracle's quantiser followed by its product -- with the
    planes read after the grid dependency, or (marked ready) before it."""
    rng = synth.rng_for(120, K)
    rows = quant_cases(rng, K)          # normal, zero, denormal, ties, huge, NaN, Inf rows
    Ns = [37, 8, 5, 64, 129, 3, 250, 17]
    entries, refs = [], []
    for i, N in enumerate(Ns):
        w = synth.ternary(rng, N, K, synth.P_ZERO)
        ws = float(synth.w_scale(w))
        planes, _ = t.trit_pack(dev(w), ws)
        x = rows[i % rows.shape[0]]
        q = torch.full((((K + 63) // 64) * 64,), 55, dtype=torch.int8, device="cuda")
        s = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
        y = torch.empty(N, dtype=torch.int32, device="cuda")
        f = torch.empty(N, dtype=torch.float32, device="cuda")
        entries.append((planes, ws, dev(x), q, s, y, f))
        q_ref, s_ref, e_ref = orc.quant(x[None, :])
        ry, rf, _ = orc.gemm(orc.pack(w), ws, q_ref, s_ref, K)
        refs.append((q_ref[0], s_ref, ry[0], rf[0], e_ref[0]))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if ready:
        torch.cuda.synchronize()   # the planes are complete before any preceding kernel
    t.trit_quant_gemv_many(t.QProjList(entries, planes_ready=ready), err)
    any_bad = any(r[4] for r in refs)
    assert int(host(err)[0]) == (t.ERR_NONFINITE if any_bad else 0)
    for (_, _, _, q, s, y, f), (q_ref, s_ref, ry, rf, _) in zip(entries, refs):
        np.testing.assert_array_equal(host(q), q_ref)
        np.testing.assert_array_equal(host(s), s_ref)
        np.testing.assert_array_equal(host(y), ry)
        assert_f32_close(host(f), rf)
        np.testing.assert_array_equal(host(f).view(np.uint32), rf.view(np.uint32))


def test_quant_gemv_many_without_code_outputs(t, orc):
    rng = synth.rng_for(121)
    K, N = 2560, 1000
    w = synth.ternary(rng, N, K, 0.45)
    x = rng.standard_normal(K).astype(np.float32)
    planes, _ = t.trit_pack(dev(w), 1.25)
    y = torch.empty(N, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t.trit_quant_gemv_many(t.QProjList([(planes, 1.25, dev(x), None, None, y, None)]), err)
    q_ref, s_ref, _ = orc.quant(x[None, :])
    ry, _, _ = orc.gemm(orc.pack(w), 1.25, q_ref, s_ref, K)
    np.testing.assert_array_equal(host(y), ry[0])


def test_quant_gemv_many_rejects_long_rows(t):
    K = t.MAX_FUSED_K + 1
    planes = torch.zeros((1, (K + 63) // 64, 16), dtype=torch.uint8, device="cuda")
    x = torch.zeros(K, dtype=torch.float32, device="cuda")
    y = torch.empty(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(t.TritError) as e:
        t.trit_quant_gemv_many(t.QProjList([(planes, 1.0, x, None, None, y, None)]), err)
    assert e.value.status == 2


# ---- tensor-core paths: weights as the 128-row operand for 17 <= M <= 128,
# ---- CTA pairs with 256 x 256 tiles above --------------------------------------

PREFILL_CASES = [(64, 33, 65), (128, 256, 64), (129, 257, 2560), (200, 300, 130), (64, 17, 6912),
                 (255, 513, 1000), (512, 6912, 2560), (320, 2560, 6912)]


@pytest.mark.parametrize("M,N,K", PREFILL_CASES)
def test_prefill_matches_oracle(t, orc, M, N, K):
    rng = synth.rng_for(130, M, N, K)
    w = synth.ternary(rng, N, K, synth.P_ZERO)
    x = padded_x(rng, M, K)
    x[:, K:] = 9                       # bytes past K are not columns
    x[0, :K] = -128
    xs = (rng.random(M) + 0.25).astype(np.float32)
    ws = float(synth.w_scale(w))
    planes, _ = t.trit_pack(dev(w), ws)
    y, f, err = t.trit_gemm(planes, ws, dev(x), dev(xs), K)
    assert int(host(err)[0]) == 0
    rows = np.arange(N) if N * M * K <= 2e8 else \
        np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 62)]))
    ry, rf, _ = orc.gemm(orc.pack(w[rows]), ws, x, xs, K)
    np.testing.assert_array_equal(host(y)[:, rows], ry)
    assert_f32_close(host(f)[:, rows], rf)
    colsum = w.astype(np.int64).sum(axis=0)
    np.testing.assert_array_equal(host(y).astype(np.int64).sum(axis=1),
                                  x[:, :K].astype(np.int64) @ colsum)


@pytest.mark.parametrize("M", [17, 200])
@pytest.mark.parametrize("K", [131071, 131072])
def test_prefill_exactness_boundary(t, orc, M, K):
    """|y| = 128*K: 16,777,088 at K = 131071 is still an exact fp32 integer on
    both tensor-core paths; K = 131072 is routed to the integer path."""
    w = np.stack([np.full(K, -1, np.int8), synth.ternary(synth.rng_for(131), 1, K, 0.4)[0]])
    x = np.zeros((M, ((K + 63) // 64) * 64), np.int8)
    x[:, :K] = -128
    x[1::2, :K] = 127
    xs = np.ones(M, np.float32)
    planes, _ = t.trit_pack(dev(w), 1.0)
    y, f, err = t.trit_gemm(planes, 1.0, dev(x), dev(xs), K)
    ry, _, _ = orc.gemm(orc.pack(w), 1.0, x, xs, K)
    assert int(ry[0, 0]) == 128 * K
    np.testing.assert_array_equal(host(y), ry)


@pytest.mark.parametrize("M", [96, 300])
def test_prefill_flags_both_set_other_rows_exact(t, orc, M):
    rng = synth.rng_for(132, M)
    N, K = 300, 2560
    w = synth.ternary(rng, N, K, synth.P_ZERO)
    p = orc.pack(w)
    for r in (3, 200, 299):
        b, k = int(rng.integers(0, p.shape[1])), int(rng.integers(0, 64))
        p[r, b, k // 8] |= 1 << (k % 8)
        p[r, b, 8 + k // 8] |= 1 << (k % 8)
    x = padded_x(rng, M, K)
    xs = np.ones(M, np.float32)
    y, f, err = t.trit_gemm(dev(p), 1.0, dev(x), dev(xs), K)
    ry, _, rerr = orc.gemm(p, 1.0, x, xs, K)
    assert int(host(err)[0]) == t.ERR_P1
    keep = rerr == 0
    assert keep.sum() == N - 3
    np.testing.assert_array_equal(host(y)[:, keep], ry[:, keep])


@pytest.mark.parametrize("M", [40, 130])
def test_prefill_outputs_optional_and_guarded(t, orc, M):
    rng = synth.rng_for(133, M)
    N, K = 250, 640
    w = synth.ternary(rng, N, K, 0.4)
    x = padded_x(rng, M, K)
    xs = (rng.random(M) + 0.5).astype(np.float32)
    planes, _ = t.trit_pack(dev(w), 0.75)
    ry, rf, _ = orc.gemm(orc.pack(w), 0.75, x, xs, K)
    g = 4096
    yb = torch.full((M * N + g,), -7, dtype=torch.int32, device="cuda")
    fb = torch.full((M * N + g,), -7.0, dtype=torch.float32, device="cuda")
    t.trit_gemm(planes, 0.75, dev(x), dev(xs), K, y_i32=yb[:M * N].view(M, N), want=())
    t.trit_gemm(planes, 0.75, dev(x), dev(xs), K, y_f32=fb[:M * N].view(M, N), want=())
    yh, fh = host(yb), host(fb)
    np.testing.assert_array_equal(yh[:M * N].reshape(M, N), ry)
    assert_f32_close(fh[:M * N].reshape(M, N), rf)
    np.testing.assert_array_equal(fh[:M * N].reshape(M, N).view(np.uint32), rf.view(np.uint32))
    assert (yh[M * N:] == -7).all() and (fh[M * N:] == -7.0).all()


# Small M on the tensor cores: every M from 13 to 128 rounds up to a multiple
# of 16 (MMA N); N ragged against the 128-row weight tiles, K against the beat.
SKINNY_CASES = [(13, 31, 191), (16, 129, 65), (17, 31, 191), (17, 129, 65), (24, 255, 2560), (32, 128, 64), (33, 9, 6912),
                (48, 1000, 640), (63, 385, 1000), (64, 6912, 2560), (100, 130, 130),
                (112, 257, 127), (127, 2560, 6912), (128, 300, 2560)]


@pytest.mark.parametrize("M,N,K", SKINNY_CASES)
def test_skinny_matches_oracle(t, orc, M, N, K):
    rng = synth.rng_for(134, M, N, K)
    w = synth.ternary(rng, N, K, synth.P_ZERO)
    x = padded_x(rng, M, K)
    x[:, K:] = -3                      # bytes past K are not columns
    x[M // 2, :K] = -128
    xs = (rng.random(M) + 0.25).astype(np.float32)
    ws = float(synth.w_scale(w))
    planes, _ = t.trit_pack(dev(w), ws)
    y, f, err = t.trit_gemm(planes, ws, dev(x), dev(xs), K)
    assert int(host(err)[0]) == 0
    rows = np.arange(N) if N * M * K <= 2e8 else \
        np.unique(np.concatenate([[0, 127, 128, N - 1], rng.integers(0, N, 60)]))
    ry, rf, _ = orc.gemm(orc.pack(w[rows]), ws, x, xs, K)
    np.testing.assert_array_equal(host(y)[:, rows], ry)
    assert_f32_close(host(f)[:, rows], rf)
    np.testing.assert_array_equal(host(f)[:, rows].view(np.uint32), rf.view(np.uint32))
    colsum = w.astype(np.int64).sum(axis=0)
    np.testing.assert_array_equal(host(y).astype(np.int64).sum(axis=1),
                                  x[:, :K].astype(np.int64) @ colsum)


def test_skinny_list_of_mixed_m(t, orc):
    """One launch over products with different M (so different MMA N and
    activation block sizes sharing one stage layout), different K and N, and
    more tiles than CTAs, mixed with products for the other paths."""
    rng = synth.rng_for(135)
    shapes = [(17, 640, 2560), (128, 300, 65), (40, 2560, 6912), (64, 1, 64), (1, 200, 640),
              (96, 6912, 2560), (8, 100, 300), (33, 129, 1000), (300, 260, 640), (20, 4000, 2560)]
    entries, refs, ws_all = [], [], []
    for M, N, K in shapes:
        w = synth.ternary(rng, N, K, float(rng.uniform(0.385, 0.508)))
        x = padded_x(rng, M, K)
        xs = (rng.random(M) + 0.5).astype(np.float32)
        ws = float(synth.w_scale(w))
        planes, _ = t.trit_pack(dev(w), ws)
        y = torch.empty((M, N), dtype=torch.int32, device="cuda")
        f = torch.empty((M, N), dtype=torch.float32, device="cuda")
        entries.append((planes, ws, dev(x), dev(xs), K, y, f))
        rows = np.arange(N) if N <= 1000 else np.unique(np.concatenate([[0, N - 1], rng.integers(0, N, 126)]))
        refs.append((rows, orc.gemm(orc.pack(w[rows]), ws, x, xs, K)))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t.trit_gemm_many(t.ProjList(entries), err)
    assert int(host(err)[0]) == 0
    for (_, _, _, _, _, y, f), (rows, (ry, rf, _)) in zip(entries, refs):
        np.testing.assert_array_equal(host(y)[:, rows], ry)
        assert_f32_close(host(f)[:, rows], rf)



def test_issue_probe_rates_are_plausible(t):
    """The issue-rate probe runs for every kind and reports a rate between one
    lane per SM-clock and the SM's 128 lanes (4 schedulers x 32 lanes) -- a
    record that is filled in and self-consistent, not a claim about the
    numbers themselves."""
    import importlib.util
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_for_probe", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    dev = torch.device("cuda", 0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    for kind in bench.ISSUE_KINDS:
        rec = t.trit_issue_probe(kind, sms * 2, 256, 64, dev)
        torch.cuda.synchronize()
        r = rec.cpu().numpy()
        assert (r[:, 2] > r[:, 1]).all(), kind
        assert set(int(v) for v in r[:, 0]) <= set(range(sms)), kind
        rates = bench.issue_rates(r, 256, 64, 64 if kind == "dp4a+lop3" else 32)
        assert 1.0 <= rates["lanes_per_clk"] <= 132.0, (kind, rates)

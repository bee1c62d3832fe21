"""GPU parity of the numerics epilogues ("Tritium ..." -- Numerics: Folded,
IntMlp) against the oracle: codes bit-exact; the IntMlp scale bit-exact (the
same double operations in the same order on both sides); the Folded scale
within 1e-6 relative (its sum of squares is reduced in a different order).
Plus one MLP chain through the C ABI: gate and up products, the integer
squared-ReLU stage, the down product -- equal to the oracle's chain."""
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


FOLDED = [(1, 1), (1, 64), (3, 65), (2, 2560), (5, 6912), (17, 6913), (33, 200)]


@pytest.mark.parametrize("M,K", FOLDED)
def test_folded_matches_oracle(t, orc, M, K):
    rng = synth.rng_for(500, M, K)
    x = (rng.standard_normal((M, K)) * rng.uniform(0.01, 100, (M, 1))).astype(np.float32)
    g = rng.uniform(0.2, 3.0, K).astype(np.float32)
    if M >= 3:
        x[1] = 0.0                                  # zero row: codes 0, scale 0
        x[2, K // 2] = np.inf                       # rejected row
    eps = 1e-5
    q, s, err = t.trit_quant_act_folded(dev(x), dev(g), eps)
    rq, rs, re = orc.quant_folded(x, g, eps)
    np.testing.assert_array_equal(host(q), rq)
    got, ref = host(s).astype(np.float64), rs.astype(np.float64)
    rel = np.where(got == ref, 0.0, np.abs(got - ref) / np.maximum(np.abs(ref), 1e-30))
    assert rel.max() <= 1e-6
    assert (int(host(err)[0]) & 8) == (8 if M >= 3 else 0)


INTMLP = [(1, 1, 100), (1, 6912, 325120), (2, 65, 2**31 - 1), (7, 2560, 40000), (17, 700, 9)]


@pytest.mark.parametrize("M,N,amp", INTMLP)
def test_intmlp_matches_oracle(t, orc, M, N, amp):
    rng = synth.rng_for(501, M, N, amp)
    ag = rng.integers(-amp, amp, size=(M, N), endpoint=True).astype(np.int64)
    au = rng.integers(-amp, amp, size=(M, N), endpoint=True).astype(np.int64)
    if M >= 2:
        ag[1] = -np.abs(ag[1]) - 1                  # all gate outputs negative: zero row
    ag = np.clip(ag, -2**31, 2**31 - 1).astype(np.int32)
    au = np.clip(au, -2**31, 2**31 - 1).astype(np.int32)
    xs = rng.uniform(0.01, 50, M).astype(np.float32)
    h, hs = t.trit_intmlp_quant(dev(ag), dev(au), 0.37, 1.9, dev(xs))
    rq, rhs = orc.intmlp_quant(ag, au, 0.37, 1.9, xs)
    np.testing.assert_array_equal(host(h), rq)
    np.testing.assert_array_equal(host(hs).view(np.int32), rhs.view(np.int32))


def test_intmlp_extremes(t, orc):
    ag = np.array([[2**31 - 1, -2**31, 1, 0, 2**31 - 1]], np.int32)
    au = np.array([[-2**31, 2**31 - 1, 1, 5, 2**31 - 1]], np.int32)
    xs = np.array([127.0], np.float32)
    h, hs = t.trit_intmlp_quant(dev(ag), dev(au), 1.0, 1.0, dev(xs))
    rq, rhs = orc.intmlp_quant(ag, au, 1.0, 1.0, xs)
    np.testing.assert_array_equal(host(h), rq)
    np.testing.assert_array_equal(host(hs).view(np.int32), rhs.view(np.int32))


def test_mlp_chain_through_the_abi(t, orc):
    """x -> folded quant -> gate, up -> IntMlp + quant -> down, every step on
    the GPU, against the same chain in the oracle (small FFN, K = 320, N = 900)."""
    rng = synth.rng_for(502)
    M, K, N = 3, 320, 900
    x = rng.standard_normal((M, K)).astype(np.float32)
    gain = rng.uniform(0.5, 1.5, K).astype(np.float32)
    Wg = synth.ternary(rng, N, K, synth.P_ZERO)
    Wu = synth.ternary(rng, N, K, synth.P_ZERO)
    Wd = synth.ternary(rng, K, N, synth.P_ZERO)
    wg, wu, wd = (float(synth.w_scale(w)) for w in (Wg, Wu, Wd))
    # oracle chain
    q, s, _ = orc.quant_folded(x, gain, 1e-5)
    yg = orc.gemm(orc.pack(Wg), wg, q, s, K)[0]
    yu = orc.gemm(orc.pack(Wu), wu, q, s, K)[0]
    hq, hs = orc.intmlp_quant(yg, yu, wg, wu, s)
    yd, yfd = orc.gemm(orc.pack(Wd), wd, hq, hs, N)[:2]
    # GPU chain (folded scale may differ in the last bit: feed the oracle's scale
    # forward only for the bit-exact comparison of the later steps' integers)
    gq, gs, gerr = t.trit_quant_act_folded(dev(x), dev(gain), 1e-5)
    np.testing.assert_array_equal(host(gq), q)
    pg, _ = t.trit_pack(dev(Wg), wg)
    pu, _ = t.trit_pack(dev(Wu), wu)
    pd, _ = t.trit_pack(dev(Wd), wd)
    s_dev = dev(s)
    g_i32 = t.trit_gemm(pg, wg, gq, s_dev, K)[0]
    u_i32 = t.trit_gemm(pu, wu, gq, s_dev, K)[0]
    np.testing.assert_array_equal(host(g_i32), yg)
    np.testing.assert_array_equal(host(u_i32), yu)
    h_i8, h_scale = t.trit_intmlp_quant(g_i32, u_i32, wg, wu, s_dev)
    np.testing.assert_array_equal(host(h_i8), hq)
    np.testing.assert_array_equal(host(h_scale).view(np.int32), hs.view(np.int32))
    d_i32, d_f32, derr = t.trit_gemm(pd, wd, h_i8, h_scale, N)
    np.testing.assert_array_equal(host(d_i32), yd)
    np.testing.assert_array_equal(host(d_f32).view(np.int32), yfd.view(np.int32))
    assert int(host(derr)[0]) == 0 and int(host(gerr)[0]) == 0


def test_div127_matches_ieee_division_on_every_float(t):
    """The dequantisation divides by 127 with a reciprocal product and one
    residual correction; over all 2^32 float bit patterns it equals the IEEE
    divide (the fp32 outputs the oracle's y_f32 formula rounds once per step)."""
    assert t.trit_check_div127() == 0


def test_intmlp_ties_and_fast_path_boundary(t, orc):
    """Exact ties (127 t / max|t| = k + 1/2) decided on both sides of the 64-bit
    path's limit max|t| < 2^56, against the oracle's exact rational rounding."""
    rows = []
    odd = [254, 1, 3, 5, 7, -1, -3, -5, 2, 127, -127, 253]
    rows.append(([1] * len(odd), odd))                              # max|t| = 254
    rows.append(([1 << 17] * len(odd), odd))                        # g^2 = 2^34: max|t| = 2^34 * 254
    g = 1 << 18                                                     # g^2 = 2^36
    rows.append(([g] * 4, [(1 << 20) - 1, 12345, -777, 1 << 19]))  # max|t| just below 2^56
    rows.append(([g] * 4, [1 << 20, 12345, -777, (1 << 19) + 1]))  # max|t| = 2^56: 128-bit path
    rows.append(([g, g], [(1 << 20) + 1, -(1 << 19) - 3]))
    for ag, au in rows:
        ag = np.array([ag], np.int32)
        au = np.array([au], np.int32)
        xs = np.array([1.7], np.float32)
        h, hs = t.trit_intmlp_quant(dev(ag), dev(au), 0.9, 1.1, dev(xs))
        rq, rhs = orc.intmlp_quant(ag, au, 0.9, 1.1, xs)
        np.testing.assert_array_equal(host(h), rq)
        np.testing.assert_array_equal(host(hs).view(np.int32), rhs.view(np.int32))


def test_intmlp_random_rows_both_paths(t, orc):
    """Many rows with magnitudes spread over 2^10 .. 2^31 (max|t| from ~2^30 to
    ~2^93), so both code paths run on many values."""
    rng = synth.rng_for(503)
    M, N = 64, 777
    amps = (2.0 ** rng.uniform(10, 31, M)).astype(np.int64)
    ag = np.stack([rng.integers(-a, a, N, endpoint=True) for a in amps])
    au = np.stack([rng.integers(-a, a, N, endpoint=True) for a in amps])
    ag = np.clip(ag, -2**31, 2**31 - 1).astype(np.int32)
    au = np.clip(au, -2**31, 2**31 - 1).astype(np.int32)
    xs = rng.uniform(0.01, 50, M).astype(np.float32)
    h, hs = t.trit_intmlp_quant(dev(ag), dev(au), 0.37, 1.9, dev(xs))
    rq, rhs = orc.intmlp_quant(ag, au, 0.37, 1.9, xs)
    np.testing.assert_array_equal(host(h), rq)
    np.testing.assert_array_equal(host(hs).view(np.int32), rhs.view(np.int32))


def _oracle_down(orc, ag, au, wg, wu, xs, Wd, wd, K):
    hq, hs = orc.intmlp_quant(ag[None, :], au[None, :], wg, wu, np.array([xs], np.float32))
    y, yf = orc.gemm(orc.pack(Wd), wd, hq, hs, K)[:2]
    return hq[0], hs[0], y[0], yf[0]


def test_mlp_chain_two_launches(t, orc):
    """x -> [gate, up] with the quantiser fused (one launch) -> [IntMlp codes +
    down product] (one launch), against the oracle's chain: every integer
    bit-exact, every fp32 bit-identical."""
    rng = synth.rng_for(504)
    K, N = 2560, 6912
    x = rng.standard_normal(K).astype(np.float32)
    Wg = synth.ternary(rng, N, K, synth.P_ZERO)
    Wu = synth.ternary(rng, N, K, synth.P_ZERO)
    Wd = synth.ternary(rng, K, N, synth.P_ZERO)
    wg, wu, wd = (float(synth.w_scale(w)) for w in (Wg, Wu, Wd))
    q, s, _ = orc.quant(x[None, :])
    ag = orc.gemm(orc.pack(Wg), wg, q, s, K)[0][0]
    au = orc.gemm(orc.pack(Wu), wu, q, s, K)[0][0]
    rh, rhs, ry, ryf = _oracle_down(orc, ag, au, wg, wu, s[0], Wd, wd, N)
    pg, _ = t.trit_pack(dev(Wg), wg)
    pu, _ = t.trit_pack(dev(Wu), wu)
    pd, _ = t.trit_pack(dev(Wd), wd)
    xd = dev(x)
    a_g = torch.empty(N, dtype=torch.int32, device="cuda")
    a_u = torch.empty(N, dtype=torch.int32, device="cuda")
    xs = torch.empty(1, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t.trit_quant_gemv_many(t.QProjList([(pg, wg, xd, None, xs, a_g, None),
                                        (pu, wu, xd, None, None, a_u, None)]), err)
    h = torch.empty(t.k_pad(N), dtype=torch.int8, device="cuda")
    hs = torch.empty(1, dtype=torch.float32, device="cuda")
    y = torch.empty(K, dtype=torch.int32, device="cuda")
    yf = torch.empty(K, dtype=torch.float32, device="cuda")
    t.trit_intmlp_gemv_many(t.MlpProjList([(pd, wd, a_g, a_u, xs, wg, wu, h, hs, y, yf)]), err)
    np.testing.assert_array_equal(host(a_g), ag)
    np.testing.assert_array_equal(host(a_u), au)
    np.testing.assert_array_equal(host(h), rh)
    np.testing.assert_array_equal(host(hs).view(np.int32), np.array([rhs]).view(np.int32))
    np.testing.assert_array_equal(host(y), ry)
    np.testing.assert_array_equal(host(yf).view(np.int32), ryf.view(np.int32))
    assert int(host(err)[0]) == 0


@pytest.mark.parametrize("K,amp", [(333, 300000), (64, 9), (6912, 2**31 - 1), (1000, 2**20)])
def test_intmlp_down_many(t, orc, K, amp):
    """Ten down projections in one call (two launches of up to eight), ragged K,
    gate/up magnitudes on both sides of the 64-bit path; one entry has a zero
    row (every gate output <= 0), one asks for no codes, scale or y_i32."""
    rng = synth.rng_for(505, K, amp)
    n_ent, N = 10, 257
    entries, want = [], []
    keep = []
    for i in range(n_ent):
        ag = rng.integers(-amp, amp, K, endpoint=True).astype(np.int64)
        au = rng.integers(-amp, amp, K, endpoint=True).astype(np.int64)
        if i == 3:
            ag = -np.abs(ag) - 1
        ag = np.clip(ag, -2**31, 2**31 - 1).astype(np.int32)
        au = np.clip(au, -2**31, 2**31 - 1).astype(np.int32)
        xs = np.float32(rng.uniform(0.5, 40))
        wg, wu = float(rng.uniform(0.5, 2)), float(rng.uniform(0.5, 2))
        Wd = synth.ternary(rng, N, K, synth.P_ZERO)
        wd = float(synth.w_scale(Wd))
        want.append(_oracle_down(orc, ag, au, wg, wu, xs, Wd, wd, K))
        pd, _ = t.trit_pack(dev(Wd), wd)
        bare = i == 5
        h = None if bare else torch.empty(t.k_pad(K), dtype=torch.int8, device="cuda")
        hs = None if bare else torch.empty(1, dtype=torch.float32, device="cuda")
        y = None if bare else torch.empty(N, dtype=torch.int32, device="cuda")
        yf = torch.empty(N, dtype=torch.float32, device="cuda")
        xsd = dev(np.array([xs], np.float32))
        entries.append((pd, wd, dev(ag), dev(au), xsd, wg, wu, h, hs, y, yf))
        keep.append((h, hs, y, yf))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t.trit_intmlp_gemv_many(t.MlpProjList(entries), err)
    for i, ((h, hs, y, yf), (rh, rhs, ry, ryf)) in enumerate(zip(keep, want)):
        np.testing.assert_array_equal(host(yf).view(np.int32), ryf.view(np.int32))
        if h is not None:
            np.testing.assert_array_equal(host(h), rh)
            np.testing.assert_array_equal(host(hs).view(np.int32), np.array([rhs]).view(np.int32))
            np.testing.assert_array_equal(host(y), ry)
        if i == 3:
            assert not ry.any() and rhs == 0
    assert int(host(err)[0]) == 0


def test_intmlp_down_rejects_bad_arguments(t):
    pd = torch.zeros((4, 2, 16), dtype=torch.uint8, device="cuda")
    a = torch.zeros(100, dtype=torch.int32, device="cuda")
    xs = torch.ones(1, dtype=torch.float32, device="cuda")
    yf = torch.empty(4, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(t.TritError):
        t.trit_intmlp_gemv_many(t.MlpProjList([(pd, 1.0, a, a, xs, 0.0, 1.0, None, None, None, yf)]), err)
    with pytest.raises(t.TritError):
        t.trit_intmlp_gemv_many(t.MlpProjList([(pd, 1.0, a, a, xs, 1.0, 1.0, None, None, None, None)]), err)

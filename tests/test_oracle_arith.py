"""Pins for the oracle's integer product, its dequantisation and its quantiser.

Independent checks used here:
  - numpy int64 dense matmul of the unpacked int8 weights (brute force);
  - the oracle's own bit-serial popcount formulation ("Tritium ..." -- On
    popcount), a second evaluation that shares no step with the int8 decode;
  - linearity in the planes: W = W+ - W-, and swapping the planes negates y;
  - the worst-case row printed on the pages ("Tritium ..." -- Defects this
    methodology found): 6912 columns of -1 against -128 gives +884,736;
  - exact rational arithmetic (fractions) for the fp32 dequantisation and the
    quantiser's rounding;
  - numpy's rint where the quantiser's multiplier is exactly 1 or 1/2;
  - invariance of the codes under a uniform power-of-two scale ("Tritium ..." --
    Numerics).
"""
from fractions import Fraction

import numpy as np
import pytest

import synth


def _rand_x(rng, M, K, lo=-128, hi=127):
    return rng.integers(lo, hi + 1, size=(M, K)).astype(np.int8)


SHAPES = [(1, 1, 1), (3, 1, 3), (17, 2, 63), (5, 3, 64), (9, 2, 65), (4, 1, 130), (33, 3, 200)]


@pytest.mark.parametrize("N,M,K", SHAPES)
def test_gemm_matches_dense_int64(orc, N, M, K):
    rng = synth.rng_for(910, N, M, K)
    w = synth.ternary(rng, N, K, 0.42)
    x = _rand_x(rng, M, K)
    x[0, 0] = -128
    p = orc.pack(w)
    ldx = ((K + 63) // 64) * 64
    xp = np.zeros((M, ldx), np.int8)
    xp[:, :K] = x
    xp[:, K:] = 77     # bytes past K are not columns and must not be read
    y, yf, err = orc.gemm(p, 1.0, xp, np.ones(M, np.float32), K)
    assert not err.any()
    want = x.astype(np.int64) @ w.astype(np.int64).T
    np.testing.assert_array_equal(y, want)


@pytest.mark.parametrize("N,M,K", SHAPES)
def test_gemm_matches_popcount_formulation(orc, N, M, K):
    rng = synth.rng_for(911, N, M, K)
    p = orc.pack(synth.ternary(rng, N, K, 0.3))
    x = _rand_x(rng, M, K)
    y, _, _ = orc.gemm(p, 1.0, x, np.ones(M, np.float32), K)
    np.testing.assert_array_equal(y, orc.gemm_popcount(p, x, K))


def test_pos_neg_split_and_plane_swap(orc):
    rng = synth.rng_for(912)
    N, M, K = 40, 2, 190
    w = synth.ternary(rng, N, K, 0.4)
    x = _rand_x(rng, M, K)
    one = np.ones(M, np.float32)
    y, _, _ = orc.gemm(orc.pack(w), 1.0, x, one, K)
    y_pos, _, _ = orc.gemm(orc.pack((w == 1).astype(np.int8)), 1.0, x, one, K)
    y_neg, _, _ = orc.gemm(orc.pack((w == -1).astype(np.int8)), 1.0, x, one, K)
    np.testing.assert_array_equal(y, y_pos - y_neg)
    p = orc.pack(w)
    swapped = np.concatenate([p[:, :, 8:], p[:, :, :8]], axis=2)
    y_sw, _, _ = orc.gemm(swapped, 1.0, x, one, K)
    np.testing.assert_array_equal(y_sw, -y)


def test_worst_case_row(orc):
    K = 6912
    p = orc.pack(np.full((1, K), -1, np.int8))
    x = np.full((1, K), -128, np.int8)
    y, _, err = orc.gemm(p, 1.0, x, np.ones(1, np.float32), K)
    assert not err.any() and int(y[0, 0]) == 884736
    assert int(orc.gemm_popcount(p, x, K)[0, 0]) == 884736


def test_row_selection_and_rejection(orc):
    rng = synth.rng_for(913)
    N, M, K = 30, 2, 130
    p = orc.pack(synth.ternary(rng, N, K, 0.42))
    x = _rand_x(rng, M, K)
    xs = np.ones(M, np.float32)
    y_all, _, _ = orc.gemm(p, 1.0, x, xs, K)
    sel = np.array([29, 0, 7, 7, 13])
    y_sel, _, err = orc.gemm(p, 1.0, x, xs, K, rows=sel)
    np.testing.assert_array_equal(y_sel, y_all[:, sel])
    bad = p.copy()
    bad[7, 1, 0] |= 4
    bad[7, 1, 8] |= 4          # both planes set at row 7, beat 1, bit 2
    y_b, _, err_b = orc.gemm(bad, 1.0, x, xs, K)
    assert err_b[7] == orc.P1 and err_b.sum() == orc.P1
    keep = np.arange(N) != 7
    np.testing.assert_array_equal(y_b[:, keep], y_all[:, keep])
    # a both-set position in the padding is an error too
    pad = p.copy()
    pad[3, 2, 7] |= 0x80
    pad[3, 2, 15] |= 0x80     # bit 63 of the last beat: column 191 >= 130
    _, _, err_p = orc.gemm(pad, 1.0, x, xs, K)
    assert err_p[3] == orc.P1


def test_output_bounded_by_support(orc):
    rng = synth.rng_for(914)
    w = synth.ternary(rng, 64, 300, 0.42)
    x = _rand_x(rng, 4, 300, -127, 127)
    y, _, _ = orc.gemm(orc.pack(w), 1.0, x, np.ones(4, np.float32), 300)
    nnz = np.count_nonzero(w, axis=1)
    assert (np.abs(y) <= 127 * nnz[None, :]).all()


def _nearest_f32(q: Fraction) -> np.float32:
    # float(q) is the correctly rounded double; for q = y * 2^s / 127 it can
    # never sit within 2^-53 of a float32 midpoint (127 is odd and its binary
    # expansion has period 7), so one more rounding to float32 is exact-nearest.
    return np.float32(float(q))


def test_dequant_power_of_two_scales(orc):
    rng = synth.rng_for(915)
    w = synth.ternary(rng, 50, 256, 0.4)
    x = _rand_x(rng, 3, 256)
    p = orc.pack(w)
    for ws_e, xs_e in [(0, 0), (-3, 5), (7, -12), (-20, 1)]:
        ws = np.float32(2.0 ** ws_e)
        xs = np.full(3, 2.0 ** xs_e, np.float32)
        y, yf, _ = orc.gemm(p, float(ws), x, xs, 256)
        for m in range(3):
            for n in range(50):
                exact = Fraction(int(y[m, n])) * Fraction(2) ** (ws_e + xs_e) / 127
                assert yf[m, n] == _nearest_f32(exact)


def test_dequant_error_bound(orc):
    rng = synth.rng_for(916)
    w = synth.ternary(rng, 80, 640, 0.42)
    x = _rand_x(rng, 2, 640)
    p = orc.pack(w)
    ws = np.float32(1.7320508)
    xs = np.array([3.14159, 0.0371], np.float32)
    y, yf, _ = orc.gemm(p, float(ws), x, xs, 640)
    u = 2.0 ** -24
    for m in range(2):
        for n in range(80):
            exact = Fraction(int(y[m, n])) * Fraction(float(ws)) * Fraction(float(xs[m])) / 127
            got = Fraction(float(yf[m, n]))
            # three roundings (two products, one quotient): |err| <= ((1+u)^3 - 1)|exact|
            assert abs(got - exact) <= Fraction(3.0001 * u) * abs(exact)
            assert (yf[m, n] == 0) == (y[m, n] == 0)


# ---- quantiser ------------------------------------------------------------

def test_quant_extremes_and_zero_row(orc):
    x = np.zeros((3, 70), np.float32)
    x[0, 5], x[0, 69] = 3.5, -3.5
    x[0, 10] = 1.0
    x[2, :] = np.linspace(-1, 0.5, 70, dtype=np.float32)
    q, s, e = orc.quant(x)
    assert q.shape == (3, 128) and not e.any()
    assert q[0, 5] == 127 and q[0, 69] == -127 and s[0] == np.float32(3.5)
    assert (q[1] == 0).all() and s[1] == 0
    assert q[2, 0] == -127 and s[2] == 1.0
    assert (q[:, 70:] == 0).all()
    assert (np.abs(q.astype(int)) <= 127).all()


def test_quant_unit_multiplier_is_rint(orc):
    """When absmax is 127 the multiplier 127/a is exactly 1 (and 1/2 at 254):
    the codes are numpy's round-half-to-even of x (of x/2)."""
    rng = synth.rng_for(917)
    base = rng.integers(-508, 509, size=(4, 300)).astype(np.float32) / 4  # quarter steps
    for amax, div in ((127.0, 1.0), (254.0, 2.0)):
        x = np.clip(base * div, -amax, amax)
        x[:, 0] = amax
        q, s, _ = orc.quant(x)
        np.testing.assert_array_equal(q[:, :300], np.rint(x / div).astype(np.int8))
        assert (s == amax).all()
    q, _, _ = orc.quant(np.array([[127.0, 2.5, 3.5, -2.5, -0.5, 0.5, 126.5]], np.float32))
    assert q[0, :7].tolist() == [127, 2, 4, -2, 0, 0, 126]


def test_quant_error_bound(orc):
    rng = synth.rng_for(918)
    x = rng.standard_normal((6, 257)).astype(np.float32)
    q, s, _ = orc.quant(x)
    for m in range(6):
        a = Fraction(float(np.abs(x[m]).max()))
        assert Fraction(float(s[m])) == a
        for c in range(257):
            exact = Fraction(float(x[m, c])) * 127 / a
            # one rounding of 127/a and one of the product sit inside the half-step
            assert abs(Fraction(int(q[m, c])) - exact) <= Fraction(1, 2) + Fraction(1, 10 ** 4)


@pytest.mark.parametrize("k", [-100, -60, -1, 1, 20, 100])
def test_quant_power_of_two_invariance(orc, k):
    rng = synth.rng_for(919, k + 200)
    x = rng.standard_normal((5, 333)).astype(np.float32) * np.float32(3.0)
    q0, s0, _ = orc.quant(x)
    xk = (x.astype(np.float64) * 2.0 ** k).astype(np.float32)
    assert np.array_equal(xk.astype(np.float64) / 2.0 ** k, x.astype(np.float64))  # exact scaling
    qk, sk, _ = orc.quant(xk)
    np.testing.assert_array_equal(qk, q0)
    np.testing.assert_array_equal(sk.astype(np.float64), s0.astype(np.float64) * 2.0 ** k)


def test_quant_rejects_non_finite_rows(orc):
    x = np.ones((4, 65), np.float32)
    x[1, 3] = np.nan
    x[3, 64] = -np.inf
    q, s, e = orc.quant(x)
    assert e.tolist() == [0, orc.NONFINITE, 0, orc.NONFINITE]
    assert (q[1] == 0).all() and (q[3] == 0).all() and s[1] == 0 and s[3] == 0
    assert (q[0, :65] == 127).all() and (q[2, :65] == 127).all()


def test_quant_denormal_row_matches_unscaled(orc):
    """A row of small integers times 2^-140 is denormal but exact; 127/absmax
    would overflow fp32 there, and the codes must still equal those of the
    unscaled integers (uniform-scale invariance)."""
    rng = synth.rng_for(920)
    n = rng.integers(-127, 128, size=(3, 200)).astype(np.float32)
    n[:, 0] = 127
    tiny = (n.astype(np.float64) * 2.0 ** -140).astype(np.float32)
    assert np.array_equal(tiny.astype(np.float64) * 2.0 ** 140, n.astype(np.float64))
    q0, s0, _ = orc.quant(n)
    qt, st, e = orc.quant(tiny)
    assert not e.any()
    np.testing.assert_array_equal(qt, q0)
    np.testing.assert_array_equal(st, tiny[:, 0])

"""Pins of the oracle's numerics epilogues ("Tritium ..." -- Numerics: Folded and
IntMlp), against closed forms, hand-built tie cases, invariants the page states
(absmax codes are unchanged by a uniform positive scale) and exact integers."""
from fractions import Fraction

import numpy as np
import pytest


# ---- IntMlp -------------------------------------------------------------------

def test_intmlp_hand_case(orc):
    # t = relu(g)^2 u = [25, 0, -28, 200]; A = 200
    q, h = orc.intmlp_quant(np.array([[5, -3, 2, 10]]), np.array([[1, 4, -7, 2]]), 0.5, 0.25,
                            [2.0])
    assert q[0, :4].tolist() == [16, 0, -18, 127]          # 15.875, 0, -17.78, 127
    assert not q[0, 4:].any()                              # zero tail to K_pad
    sg, su = 0.5 * 2.0 / 127, 0.25 * 2.0 / 127
    assert h[0] == np.float32(200 * (sg * sg) * su)


def test_intmlp_ties_round_to_even(orc):
    # A = 254 (g = 1, u = 254); t = u for g = 1, so code = round(u / 2)
    u = np.array([[254, 1, 3, 5, 7, -1, -3, -5, 2]])
    g = np.ones_like(u)
    q, _ = orc.intmlp_quant(g, u, 1.0, 1.0, [1.0])
    assert q[0, :9].tolist() == [127, 0, 2, 2, 4, 0, -2, -2, 1]


def test_intmlp_relu_and_zero_row(orc):
    q, h = orc.intmlp_quant(np.array([[-1, -7, 0, -100]]), np.array([[9, 9, 9, 9]]), 1.0, 1.0,
                            [3.0])
    assert not q.any() and h[0] == 0.0


def test_intmlp_invariants(orc):
    rng = np.random.default_rng(5)
    for _ in range(20):
        N = int(rng.integers(1, 300))
        g = rng.integers(-3000, 3000, size=(2, N)).astype(np.int32)
        u = rng.integers(-3000, 3000, size=(2, N)).astype(np.int32)
        q, h = orc.intmlp_quant(g, u, 0.7, 1.3, [0.5, 2.0])
        t = np.maximum(g.astype(np.int64), 0) ** 2 * u.astype(np.int64)
        for m in range(2):
            A = np.abs(t[m]).max()
            if A == 0:
                assert not q[m].any()
                continue
            # the largest |t| maps to +-127; signs follow t; |q| <= 127
            i = int(np.abs(t[m]).argmax())
            assert abs(int(q[m, i])) == 127 and np.sign(q[m, i]) == np.sign(t[m, i])
            assert (np.sign(q[m, :N]) * np.sign(t[m]) >= 0).all()
        # negating the up output negates every code; scaling it by 3 keeps them
        qn, _ = orc.intmlp_quant(g, -u, 0.7, 1.3, [0.5, 2.0])
        assert (qn == -q).all()
        if np.abs(u).max() * 3 < 2**31:
            q3, h3 = orc.intmlp_quant(g, 3 * u, 0.7, 1.3, [0.5, 2.0])
            assert (q3 == q).all()
            assert np.allclose(h3, 3 * h, rtol=1e-6)


def test_intmlp_page_bound_and_past_int64(orc):
    # [TRI] Numerics: |t| < 2^55 for a 2560-column projection: |a| <= 127 * 2560
    a = 127 * 2560
    g = np.array([[a, a, 1000, -5]], np.int32)
    u = np.array([[a, -a, 77, 3]], np.int32)
    q, _ = orc.intmlp_quant(g, u, 1.0, 1.0, [1.0])
    t = [a * a * a, -a * a * a, 1000 * 1000 * 77, 0]
    assert abs(t[0]) < 2**55
    want = [int(round(Fraction(127 * v, t[0]))) for v in t]      # Fraction rounds half to even
    assert q[0, :4].tolist() == want
    # past int64: 2^31-1 squared times -2^31 is about -2^93; still exact
    g = np.array([[2**31 - 1, 2**20]], np.int32)
    u = np.array([[-2**31, 2**31 - 1]], np.int32)
    q, h = orc.intmlp_quant(g, u, 1.0, 1.0, [127.0])
    A = (2**31 - 1) ** 2 * 2**31
    t1 = 2**40 * (2**31 - 1)
    assert q[0, :2].tolist() == [-127, int(round(Fraction(127 * t1, A)))]
    hi, lo = A >> 64, A & (2**64 - 1)
    assert h[0] == np.float32((float(hi) * 2.0**64 + float(lo)) * 1.0)   # S_g = S_u = 1


def test_intmlp_exact_rational_on_random_rows(orc):
    rng = np.random.default_rng(11)
    g = rng.integers(-50000, 50000, size=(3, 200)).astype(np.int32)
    u = rng.integers(-50000, 50000, size=(3, 200)).astype(np.int32)
    q, _ = orc.intmlp_quant(g, u, 1.0, 1.0, [1.0, 1.0, 1.0])
    for m in range(3):
        t = [max(int(a), 0) ** 2 * int(b) for a, b in zip(g[m], u[m])]
        A = max(abs(v) for v in t)
        assert q[m, :200].tolist() == [int(round(Fraction(127 * v, A))) for v in t]


# ---- Folded ---------------------------------------------------------------------

def test_folded_equals_plain_quant_when_gain_is_one(orc):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 333)).astype(np.float32)
    q, s, e = orc.quant_folded(x, np.ones(333, np.float32), 1e-5)
    q0, s0, e0 = orc.quant(x)
    assert (q == q0).all() and (e == 0).all()
    rms = np.sqrt((x.astype(np.float64) ** 2).mean(1) + 1e-5)
    assert np.allclose(s, s0 / rms, rtol=1e-6)


@pytest.mark.parametrize("k", [-3, 0, 1, 5])
def test_folded_matches_the_materialised_path_at_power_of_two_rms(orc, k):
    """Reference mode normalises, then quantises; Folded quantises x (.) g and
    divides the scale by the rms.  With a power-of-two rms the normalisation is
    exact in fp32, so both give the same codes and the same scale."""
    rng = np.random.default_rng(17 + k)
    K = 256
    # rows whose mean square is exactly 4^k: +-2^k at every column
    x = (rng.choice([-1.0, 1.0], size=(3, K)) * 2.0**k).astype(np.float32)
    x[:, ::7] *= 0                       # zeros change the mean: compensate with eps
    ms = (x.astype(np.float64) ** 2).mean(1)
    assert (ms == ms[0]).all()
    eps = 4.0**k - ms[0]                 # mean + eps = 4^k exactly
    g = rng.uniform(0.5, 2.0, K).astype(np.float32)
    q, s, e = orc.quant_folded(x, g, eps)
    y = (x / np.float32(2.0**k)) * g     # the materialised, normalised row (exact division)
    q1, s1, e1 = orc.quant(y)
    assert (q == q1).all() and (s == s1).all() and not e.any()


def test_folded_rejects_non_finite(orc):
    x = np.ones((3, 64), np.float32)
    g = np.ones(64, np.float32)
    x[0, 5] = np.nan
    x[1, 0] = 3e38
    g2 = g.copy()
    g2[0] = 10.0                         # 3e38 * 10 overflows to inf in fp32
    q, s, e = orc.quant_folded(x, g2, 1e-5)
    assert e[0] == 8 and e[1] == 8 and e[2] == 0
    assert not q[:2].any() and s[0] == 0 and s[1] == 0

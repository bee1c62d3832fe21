"""The fp32 estimate behind every IntMlp code on the GPU, emulated on the host
with numpy float32 (each operation rounded once, as the kernels' __fmul_rn /
__fadd_rn / conversions do): p = fl(fl(fl(g)^2) * fl(|u|)) * fl(127 / fl(A))
stays within 7.6e-5 of the exact 127|t|/A, so wherever p is further than the
kernels' threshold from a half-integer its round-half-even equals the exact
code round-half-even(127|t|/A) ("Tritium ..." -- Numerics, IntMlp).  CPU only."""
import numpy as np

F32 = np.float32


def fl_A(A: int) -> np.float32:
    """fl(A) as the kernels form it: fl(hi) * 2^64 + fl(lo), fp32."""
    hi, lo = A >> 64, A & ((1 << 64) - 1)
    return F32(F32(hi) * F32(2.0 ** 64)) + F32(lo)


def estimate(ag: int, au: int, kf: np.float32) -> np.float32:
    g = F32(max(ag, 0))
    tf = F32(F32(g * g) * F32(abs(au)))
    return F32(tf * kf)


def exact_code(t: int, A: int) -> int:
    """round-half-even(127 t / A) for 0 <= t <= A, A > 0, in integers."""
    n, d = 127 * t, A
    q, r = divmod(n, d)
    if 2 * r > d or (2 * r == d and q % 2):
        q += 1
    return q


def rne_magic(p: np.float32):
    """The kernels' rounding: p + 1.5 * 2^23 - 1.5 * 2^23 (fp32), and the
    remainder p - that integer."""
    big = F32(p + F32(12582912.0))
    r = F32(big - F32(12582912.0))
    return int(r), F32(p - r)


def samples(rng, n):
    out = []
    for _ in range(n):
        bits = int(rng.integers(1, 32))
        ag = int(rng.integers(-(1 << bits), 1 << bits))
        au = int(rng.integers(-(1 << bits), 1 << bits))
        out.append((ag, au))
    return out


def test_estimate_within_bound_and_codes_exact_off_ties():
    rng = np.random.default_rng(20251202)
    checked = near = 0
    for _row in range(60):
        cols = samples(rng, 400)
        ts = [max(ag, 0) ** 2 * abs(au) for ag, au in cols]
        A = max(ts)
        if A == 0:
            continue
        kf = F32(F32(127.0) / fl_A(A))
        for (ag, au), t in zip(cols, ts):
            p = estimate(ag, au, kf)
            exact = 127 * t / A
            assert abs(float(p) - exact) < 7.6e-5, (ag, au, A)
            q, fr = rne_magic(p)
            if abs(float(fr)) < 0.49985:
                assert min(q, 127) == exact_code(t, A), (ag, au, A)
                checked += 1
            else:
                near += 1
    assert checked > 20000 and near < checked // 100


def test_extremes_of_the_int32_range():
    """|a_g| and |a_u| at 2^31 - 1 (t near 2^93, the 128-bit range) and a row
    whose maximum is the single largest column."""
    big = (1 << 31) - 1
    cols = [(big, big), (big, -big), (big, 1), (1, big), (-big, big), (big // 3, -(big // 5)),
            (46341, 2), (3, 3), (0, big)]
    ts = [max(ag, 0) ** 2 * abs(au) for ag, au in cols]
    A = max(ts)
    kf = F32(F32(127.0) / fl_A(A))
    for (ag, au), t in zip(cols, ts):
        p = estimate(ag, au, kf)
        assert abs(float(p) - 127 * t / A) < 7.6e-5
        q, fr = rne_magic(p)
        if abs(float(fr)) < 0.49985:
            assert min(q, 127) == exact_code(t, A)


def test_magic_rounding_is_round_half_even():
    for p in (0.0, 0.5, 1.5, 2.5, 126.5, 127.0, 0.49999997, 63.75, 100.25):
        q, fr = rne_magic(F32(p))
        assert q == round(p)   # Python's round is half-to-even
        assert float(fr) == float(F32(p)) - q

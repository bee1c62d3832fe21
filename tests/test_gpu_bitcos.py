"""GPU parity of the BITCOS product (trit_bitcos_gemv_many) with the oracle
("BITCOS: Intel's Ternary LLM Weight Format Goes Below 1.58 Bits" -- A bitmap
and a sign): exact int32 and identical fp32 bits, element by element, on
shapes that span several warps' rows and ragged K and N; the 30-layer stack on
sampled rows; and bit identity with the 2-bit plane path on the same W."""
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


def host(x):
    torch.cuda.synchronize()
    return x.cpu().numpy()


def product(t, orc, N, K, p0, seed, rows=None):
    rng = synth.rng_for(740, N, K, seed)
    w = synth.ternary(rng, N, K, p0)
    kp = ((K + 63) // 64) * 64
    x = rng.integers(-128, 128, size=kp).astype(np.int8)
    x[K:] = rng.integers(-128, 128, size=kp - K)          # bytes past K are not columns
    x[: min(K, 3)] = -128
    xs = np.float32(rng.random() + 0.05)
    ws = float(synth.w_scale(w)) if p0 < 1.0 else 1.0
    W = t.BitcosWeights(*t.trit_bitcos_pack(w), K)
    xd = torch.from_numpy(x).cuda()
    xsd = torch.tensor([xs], dtype=torch.float32, device="cuda")
    y = torch.full((N,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    f = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
    ref = orc.bitcos_gemv(*orc.bitcos_pack_blocked(w), K, ws, x, float(xs), rows=rows)
    return (W, ws, xd, xsd, y, f), ref, w, x, xs


SHAPES = [(1, 1, 0.42), (3, 63, 0.42), (9, 64, 0.0), (9, 64, 1.0), (31, 65, 0.5), (100, 130, 0.3),
          (257, 2560, 0.42), (640, 2560, 0.508), (1000, 6912, 0.385), (129, 6913, 0.42),
          (40, 16384, 0.42)]


@pytest.mark.parametrize("N,K,p0", SHAPES)
def test_bitcos_gemv_matches_oracle(t, orc, N, K, p0):
    e, (ry, rf), *_ = product(t, orc, N, K, p0, 0)
    t.trit_bitcos_gemv_many(t.BitcosList([e]))
    np.testing.assert_array_equal(host(e[4]), ry)
    np.testing.assert_array_equal(host(e[5]).view(np.uint32), rf.view(np.uint32))


def test_bitcos_list_of_mixed_products_and_optional_outputs(t, orc):
    shapes = [(300, 2560, 0.42), (7, 65, 0.5), (2560, 6912, 0.4), (64, 640, 0.45), (1, 3, 0.0)]
    ents, refs = [], []
    for i, (N, K, p0) in enumerate(shapes):
        e, ref, *_ = product(t, orc, N, K, p0, i + 1)
        W, ws, xd, xsd, y, f = e
        if i == 1:
            f = None
        if i == 3:
            y = None
        ents.append((W, ws, xd, xsd, y, f))
        refs.append(ref)
    t.trit_bitcos_gemv_many(t.BitcosList(ents))
    for (W, ws, xd, xsd, y, f), (ry, rf) in zip(ents, refs):
        if y is not None:
            np.testing.assert_array_equal(host(y), ry)
        if f is not None:
            np.testing.assert_array_equal(host(f).view(np.uint32), rf.view(np.uint32))


def test_bitcos_equals_plane_path(t, orc):
    """Same W, same x: the BITCOS product and trit_gemv give identical bits."""
    (W, ws, xd, xsd, y, f), _, w, x, xs = product(t, orc, 2560, 6912, 0.42, 9)
    t.trit_bitcos_gemv_many(t.BitcosList([(W, ws, xd, xsd, y, f)]))
    planes, _ = t.trit_pack(torch.from_numpy(w).cuda(), ws)
    y2, f2, err = t.trit_gemv(planes, ws, xd, float(np.asarray(xs).reshape(-1)[0]), 6912)
    assert int(host(err)[0]) == 0
    np.testing.assert_array_equal(host(y), host(y2).reshape(-1))
    np.testing.assert_array_equal(host(f).view(np.uint32), host(f2).reshape(-1).view(np.uint32))


def test_bitcos_stack_sampled(t, orc):
    """The 30-layer stack (210 products) in one call; sampled rows of every
    13th product against the oracle."""
    items = list(synth.stack_items(synth.LAYERS))
    ents, checks = [], []
    for i, (layer, idx, name, N, K) in enumerate(items):
        w = synth.stack_weights(6, layer, idx)
        ws = float(synth.w_scale(w))
        x = synth.projection_acts(6, layer, idx, 1)
        q = np.zeros(((K + 63) // 64) * 64, np.int8)
        q[:K] = np.clip(np.rint(x[0, :K] * (127 / max(np.abs(x[0, :K]).max(), 1e-30))), -127, 127)
        W = t.BitcosWeights(*t.trit_bitcos_pack(w), K)
        xd = torch.from_numpy(q).cuda()
        xsd = torch.tensor([0.5], dtype=torch.float32, device="cuda")
        y = torch.empty(N, dtype=torch.int32, device="cuda")
        f = torch.empty(N, dtype=torch.float32, device="cuda")
        ents.append((W, ws, xd, xsd, y, f))
        if i % 13 == 0:
            rows = np.unique(np.concatenate([[0, N - 1], synth.rng_for(741, i).integers(0, N, 40)]))
            checks.append((i, rows, orc.bitcos_gemv(*orc.bitcos_pack_blocked(w), K, ws, q, 0.5,
                                                    rows=rows)))
    t.trit_bitcos_gemv_many(t.BitcosList(ents))
    for i, rows, (ry, rf) in checks:
        np.testing.assert_array_equal(host(ents[i][4])[rows], ry)
        np.testing.assert_array_equal(host(ents[i][5])[rows].view(np.uint32), rf.view(np.uint32))

"""GPU parity of the batch-1 MLP block in two launches (trit_mlp_gate_up, then
trit_mlp_down; "Tritium ..." -- Numerics, IntMlp) against the oracle's chain:
quantise x, gate and up products, the integer squared-ReLU stage with its
codes and scale, the down product.  Every output -- x_scale, a_gate, a_up,
h_i8, h_scale, y_i32, y_f32 -- bit-identical, on the pre-loading path (gate
and up paired in one launch that publishes max|t| partials; the down launch
reduces them) and on the fused fallback for rows longer than it takes."""
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


def make_block(t, rng, K, F, N, outs=True, x=None, w_gate=None):
    Wg = synth.ternary(rng, F, K, float(rng.uniform(0.385, 0.508))) if w_gate is None else w_gate
    Wu = synth.ternary(rng, F, K, float(rng.uniform(0.385, 0.508)))
    Wd = synth.ternary(rng, N, F, float(rng.uniform(0.385, 0.508)))
    ws = [float(synth.w_scale(w)) for w in (Wg, Wu, Wd)]
    P = [t.trit_pack(dev(w), s)[0] for w, s in zip((Wg, Wu, Wd), ws)]
    if x is None:
        x = rng.standard_normal(K).astype(np.float32)
    cuda = dict(device="cuda")
    bufs = dict(
        x=dev(x), x_scale=torch.full((1,), -1.0, dtype=torch.float32, **cuda),
        a_gate=torch.full((F,), 7, dtype=torch.int32, **cuda),
        a_up=torch.full((F,), 7, dtype=torch.int32, **cuda),
        tmax=torch.full((t.trit_mlp_tmax_bytes(F),), 0xAB, dtype=torch.uint8, **cuda),
        h_i8=torch.full((t.k_pad(F),), 55, dtype=torch.int8, **cuda) if outs else None,
        h_scale=torch.full((1,), -1.0, dtype=torch.float32, **cuda) if outs else None,
        y_i32=torch.full((N,), 3, dtype=torch.int32, **cuda),
        y_f32=torch.full((N,), 3.0, dtype=torch.float32, **cuda))
    entry = (P[0], P[1], P[2], ws[0], ws[1], ws[2], bufs["x"], bufs["x_scale"], bufs["a_gate"],
             bufs["a_up"], bufs["tmax"], bufs["h_i8"], bufs["h_scale"], bufs["y_i32"], bufs["y_f32"])
    return entry, bufs, (Wg, Wu, Wd, ws, x)


def oracle_block(orc, ref, K, F):
    Wg, Wu, Wd, ws, x = ref
    q, s, e = orc.quant(x[None, :])
    assert not e.any()
    ag, _, _ = orc.gemm(orc.pack(Wg), ws[0], q, s, K)
    au, _, _ = orc.gemm(orc.pack(Wu), ws[1], q, s, K)
    h, hs = orc.intmlp_quant(ag, au, ws[0], ws[1], s)
    y, f, err = orc.gemm(orc.pack(Wd), ws[2], h, hs, F)
    assert not err.any()
    return dict(x_scale=s, a_gate=ag[0], a_up=au[0], h_i8=h[0], h_scale=hs, y_i32=y[0], y_f32=f[0])


def check(bufs, ref):
    for k, v in ref.items():
        if bufs[k] is None:
            continue
        got = host(bufs[k])
        if v.dtype == np.float32:
            np.testing.assert_array_equal(got.view(np.uint32), v.view(np.uint32), err_msg=k)
        else:
            np.testing.assert_array_equal(got, v, err_msg=k)


def run(t, blocks, ready):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if ready:
        torch.cuda.synchronize()   # the planes are complete before any preceding kernel
    bl = t.MlpBlockList([b[0] for b in blocks], planes_ready=ready)
    t.trit_mlp_gate_up(bl, err)
    t.trit_mlp_down(bl, err)
    assert int(host(err)[0]) == 0


SHAPES = [(2560, 6912, 2560), (100, 77, 33), (640, 1000, 129), (13312, 300, 64),
          (13376, 64, 16), (64, 8960, 24), (256, 9024, 40), (1, 1, 1), (65, 31, 9)]


@pytest.mark.parametrize("ready", [False, True])
@pytest.mark.parametrize("K,F,N", SHAPES)
def test_mlp_block_matches_oracle(t, orc, K, F, N, ready):
    """One block per call; the pre-loading kernel takes gate/up rows of up to
    13,312 columns and down rows (F) of up to 8,960, and 13,376 / 9,024 go
    through the fused fallback."""
    rng = synth.rng_for(140, K, F, N, int(ready))
    blk = make_block(t, rng, K, F, N)
    run(t, [blk], ready)
    check(blk[1], oracle_block(orc, blk[2], K, F))


def test_mlp_blocks_in_one_call(t, orc):
    """Thirty-four blocks in one call (five launches of at most eight pairs each),
    mixed shapes, one past the pre-loading limit, some without h outputs;
    repeated so the partials of a second token overwrite the first."""
    rng = synth.rng_for(141)
    shapes = [(2560, 6912, 2560), (2560, 2560, 640), (128, 200, 300), (13376, 64, 16),
              (640, 96, 8), (200, 33, 65), (2560, 6912, 2560), (64, 64, 64), (320, 1111, 77)]
    shapes += [(64 + 64 * (i % 3), 40 + i, 24) for i in range(25)]
    blocks = [make_block(t, rng, K, F, N, outs=(i % 3 != 1)) for i, (K, F, N) in enumerate(shapes)]
    for rep in range(2):
        if rep:
            for b in blocks:   # a new token: new rows
                b[1]["x"].copy_(dev(rng.standard_normal(b[1]["x"].numel()).astype(np.float32)))
        run(t, blocks, rep == 1)
        for b, (K, F, N) in zip(blocks, shapes):
            Wg, Wu, Wd, ws, _ = b[2]
            ref = oracle_block(orc, (Wg, Wu, Wd, ws, host(b[1]["x"])), K, F)
            check(b[1], ref)


def test_mlp_block_degenerate_rows(t, orc):
    """A zero input row (every code and scale 0) and a block whose gate
    outputs are all <= 0 (relu leaves t = 0 everywhere: max|t| = 0, codes 0,
    h_scale 0, y 0)."""
    rng = synth.rng_for(142)
    K, F, N = 640, 200, 72
    zero = make_block(t, rng, K, F, N, x=np.zeros(K, dtype=np.float32))
    neg = make_block(t, rng, K, F, N, x=np.abs(rng.standard_normal(K)).astype(np.float32) + 0.1,
                     w_gate=-np.ones((F, K), dtype=np.int8))
    run(t, [zero, neg], True)
    for b in (zero, neg):
        ref = oracle_block(orc, b[2], K, F)
        check(b[1], ref)
        assert not host(b[1]["h_i8"]).any()
        assert float(host(b[1]["h_scale"])[0]) == 0.0
    assert (host(neg[1]["a_gate"]) <= 0).all()


def test_mlp_block_rejects_planes_that_do_not_chain(t):
    rng = synth.rng_for(143)
    blk = make_block(t, rng, 128, 64, 32)
    e = list(blk[0])
    e[2] = torch.zeros((32, 2, 16), dtype=torch.uint8, device="cuda")   # down planes of K = 128
    with pytest.raises(ValueError):
        t.MlpBlockList([tuple(e)])

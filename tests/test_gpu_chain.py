"""The dependency-ordered decode (LayerChain): two layers of the BitNet-shaped
stack, four launches per layer (five with the IntMlp quantiser as a launch of
its own), each reading the previous launch's outputs,
against the oracle's chain -- quantiser, product, quantiser of the product's
fp32 output, ..., IntMlp quantiser, down product -- every int32 output
bit-exact and every fp32 output bit-identical at every stage (so the chain
stays exact however many stages it has)."""
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


@pytest.mark.parametrize("mlp_form", ["paired", "split", "fused"])
def test_layer_chain_matches_oracle_chain(t, orc, mlp_form):
    from bit_plane_select_gb300.stack import LayerChain
    seed, layers = 9, 2
    names = [p[0] for p in synth.PROJECTIONS]
    W = [{n: synth.stack_weights(seed, layer, i) for i, n in enumerate(names)} for layer in range(layers)]
    ws = [{n: float(synth.w_scale(W[l][n])) for n in names} for l in range(layers)]
    chain = LayerChain([{n: (torch.from_numpy(W[l][n]), ws[l][n]) for n in names} for l in range(layers)],
                       mlp_form=mlp_form)
    assert chain.launches_per_step == (5 if mlp_form == "split" else 4) * layers
    xs = [synth.projection_acts(seed, l, 0, 1)[0] for l in range(layers)]
    for l in range(layers):
        chain.x[l].copy_(torch.from_numpy(xs[l]))
    for _ in range(2):         # repeated tokens give the same outputs
        chain.step()
    assert int(host(chain.err)[0]) == 0
    check_chain_against_oracle(orc, chain, W, ws, xs, layers)


def check_chain_against_oracle(orc, chain, W, ws, xs, layers):

    def prod(name, l, x_f32):
        q, s, e = orc.quant(x_f32[None, :])
        assert not e.any()
        w = W[l][name]
        y, f, err = orc.gemm(orc.pack(w), ws[l][name], q, s, w.shape[1])
        assert not err.any()
        return y[0], f[0], s

    for l in range(layers):
        L = chain.layers[l]
        outs = {}
        for n in ("q", "k", "v"):
            outs[n] = prod(n, l, xs[l])
        outs["o"] = prod("o", l, outs["q"][1])
        outs["gate"] = prod("gate", l, outs["o"][1])
        outs["up"] = prod("up", l, outs["o"][1])
        s_gu = outs["gate"][2]
        h, hs = orc.intmlp_quant(outs["gate"][0][None, :], outs["up"][0][None, :],
                                 ws[l]["gate"], ws[l]["up"], s_gu)
        Wd = W[l]["down"]
        yd, fd, err = orc.gemm(orc.pack(Wd), ws[l]["down"], h, hs, Wd.shape[1])
        assert not err.any()
        for n in ("q", "k", "v", "o"):
            np.testing.assert_array_equal(host(L["y_" + n]), outs[n][0])
            np.testing.assert_array_equal(host(L["f_" + n]).view(np.uint32), outs[n][1].view(np.uint32))
        np.testing.assert_array_equal(host(L["a_gate"]), outs["gate"][0])
        np.testing.assert_array_equal(host(L["a_up"]), outs["up"][0])
        np.testing.assert_array_equal(host(L["s_gu"]).view(np.uint32), s_gu.view(np.uint32))
        if chain.mlp_form == "split":   # the IntMlp codes and scale the down product read
            np.testing.assert_array_equal(host(L["h"])[:h.shape[1]], h[0])
            np.testing.assert_array_equal(host(L["s_h"]).view(np.uint32), hs.view(np.uint32))
        np.testing.assert_array_equal(host(L["y_down"]), yd[0])
        np.testing.assert_array_equal(host(L["f_down"]).view(np.uint32), fd[0].view(np.uint32))


def test_layer_chain_rejects_shapes_that_do_not_chain(t):
    from bit_plane_select_gb300.stack import LayerChain
    z = lambda n, k: (torch.zeros((n, k), dtype=torch.int8), 1.0)
    bad = {"q": z(64, 64), "k": z(16, 64), "v": z(16, 64), "o": z(64, 128), "gate": z(96, 64),
           "up": z(96, 64), "down": z(64, 96)}
    with pytest.raises(ValueError):
        LayerChain([bad])


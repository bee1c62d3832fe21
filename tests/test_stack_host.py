"""Host-side checks of the runtime classes that need no GPU: argument
validation that happens before any device work."""
import pytest

torch = pytest.importorskip("torch")


def test_layer_chain_rejects_unknown_mlp_form():
    from bit_plane_select_gb300.stack import LayerChain
    with pytest.raises(ValueError):
        LayerChain([], device="cpu", mlp_form="unrolled")
    assert LayerChain.MLP_FORMS == ("paired", "split", "fused")


def test_mlp_block_list_checks_that_the_planes_chain():
    import bit_plane_select_gb300 as t
    K, F, N = 128, 64, 32
    planes = lambda rows, k: torch.zeros((rows, (k + 63) // 64, 16), dtype=torch.uint8)
    x = torch.zeros(K)
    buf = lambda n, dt: torch.zeros(n, dtype=dt)
    good = [planes(F, K), planes(F, K), planes(N, F), 1.0, 1.0, 1.0, x, buf(1, torch.float32),
            buf(F, torch.int32), buf(F, torch.int32), buf(64, torch.uint8), None, None,
            buf(N, torch.int32), None]
    for i, bad in ((1, planes(F + 8, K)), (2, planes(N, K)), (0, planes(F, 2 * K))):
        e = list(good)
        e[i] = bad
        with pytest.raises(ValueError):
            t.MlpBlockList([tuple(e)])
    with pytest.raises(ValueError):   # host tensors are refused after the shape check
        t.MlpBlockList([tuple(good)])

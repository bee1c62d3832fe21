"""A .trit v1 file straight to the device: the library's reader maps the file,
uploads a ternary tensor's bytes unchanged, and the products over the uploaded
planes equal the oracle's products over the planes the oracle packed itself."""
import numpy as np
import pytest

import synth
from oracle import container as C
from test_container import trit_payload, write_file

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


def test_file_upload_then_gemv_matches_oracle(t, orc, tmp_path):
    from bit_plane_select_gb300.trit_file import TritFile
    rng = synth.rng_for(400)
    N, K = 640, 2560
    w = synth.ternary(rng, N, K, synth.P_ZERO)
    ws = float(synth.w_scale(w))
    planes_host = orc.pack(w)                       # the oracle's packing
    small = synth.ternary(rng, 3, 70, 0.3)
    dense = rng.standard_normal(24).astype(np.float32)
    data = write_file([
        dict(name="blk.0.attn_k.weight", dtype=1, dims=[N, K], scale=ws,
             payload=planes_host.tobytes()),
        dict(name="blk.0.norm", dtype=0, dims=[24], scale=1.0, payload=dense.tobytes()),
        dict(name="tiny", dtype=1, dims=[3, 70], scale=1.0, payload=trit_payload(small)),
    ])
    assert C.first_violation(data)[0] == 0
    path = tmp_path / "model.trit"
    path.write_bytes(data)
    with TritFile.open(str(path)) as f:
        f.verify()
        info = f.tensor(f.find("blk.0.attn_k.weight"))
        assert info["scale"] == np.float32(ws)
        planes = f.upload("blk.0.attn_k.weight")
        tiny = f.upload("tiny")
        torch.cuda.synchronize()
    np.testing.assert_array_equal(planes.cpu().numpy().reshape(-1), planes_host.reshape(-1))
    # the uploaded planes pass the device check and unpack to the weights
    err, first = t.trit_verify(planes, K)
    assert int(err.item()) == 0
    back, _ = t.trit_unpack(tiny, 70)
    np.testing.assert_array_equal(back.cpu().numpy(), small)
    # products over the uploaded planes
    x = synth.activations(rng, 1, K)
    q, s, _ = orc.quant(x)
    y, fy, err = t.trit_gemv(planes, ws, torch.from_numpy(q).cuda(), float(s.reshape(-1)[0]), K)
    ry, rf = orc.gemm(planes_host, ws, q, s, K)[:2]
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(y.cpu().numpy(), ry.reshape(-1))
    np.testing.assert_array_equal(fy.cpu().numpy().view(np.int32), rf.reshape(-1).view(np.int32))

"""The library's BITCOS packer (host code, no GPU) against the oracle's
blocked form ("BITCOS: Intel's Ternary LLM Weight Format Goes Below 1.58
Bits" -- A bitmap and a sign), and its argument checks."""
import ctypes

import numpy as np
import pytest

import oracle
import synth


@pytest.fixture(scope="module")
def trit():
    from bit_plane_select_gb300 import build
    build.build()
    import bit_plane_select_gb300 as t
    return t


SHAPES = [(1, 1, 0.5), (3, 63, 0.42), (4, 64, 0.0), (4, 64, 1.0), (7, 65, 0.42), (33, 130, 0.3),
          (17, 2560, 0.5), (5, 6913, 0.385), (2, 16384, 0.42)]


@pytest.mark.parametrize("N,K,p0", SHAPES)
def test_packer_matches_oracle(trit, N, K, p0):
    w = synth.ternary(synth.rng_for(720, N, K, int(100 * p0)), N, K, p0)
    got = trit.trit_bitcos_pack(w)
    ref = oracle.bitcos_pack_blocked(w)
    for g, r in zip(got, ref):
        np.testing.assert_array_equal(g, r)


def test_size_query_and_rejections(trit):
    L = trit.lib()
    w = np.array([[1, 0, -1], [0, 0, 0]], np.int8)
    words = ctypes.c_int64(-1)
    wp = ctypes.c_void_p(w.ctypes.data)
    assert L.trit_bitcos_pack(wp, 2, 3, None, None, None, ctypes.byref(words)) == 0
    assert words.value == 1 + 0 + 2          # ceil(2/32) + ceil(0/32) + 2 guard words
    assert L.trit_bitcos_pack(None, 2, 3, None, None, None, ctypes.byref(words)) == 1
    assert L.trit_bitcos_pack(wp, 2, 3, None, None, None, None) == 1
    buf = (ctypes.c_uint32 * 8)()
    assert L.trit_bitcos_pack(wp, 2, 3, None, None, buf, ctypes.byref(words)) == 1
    assert L.trit_bitcos_pack(wp, 0, 3, None, None, None, ctypes.byref(words)) == 2
    assert L.trit_bitcos_pack(wp, 2, trit.BITCOS_MAX_K + 1, None, None, None,
                              ctypes.byref(words)) == 2
    bad = np.array([[1, 0, -2]], np.int8)
    with pytest.raises(trit.TritError) as e:
        trit.trit_bitcos_pack(bad)
    assert e.value.status == 9

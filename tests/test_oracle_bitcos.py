"""Pins for the oracle's BITCOS functions ("BITCOS: Intel's Ternary LLM Weight
Format Goes Below 1.58 Bits" -- A bitmap and a sign), against things other than
the oracle itself:
  - numpy's packbits (little bit order) of the presence and sign indicators;
  - the page's round-trip assertion, on edge sizes;
  - the page's printed packed sizes for two tensors (tests/golden);
  - the flat layout, for the blocked layout's rows;
  - the independent bit-plane oracle (oracle.gemm), for the BITCOS product.
"""
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def ternary(rng, n, p0):
    return synth.ternary(rng, 1, n, p0)[0]


@pytest.mark.parametrize("n", [0, 1, 7, 8, 9, 63, 64, 65, 1000, 4099])
@pytest.mark.parametrize("p0", [0.0, 0.42, 1.0])
def test_flat_layout_is_packbits_of_presence_and_sign(n, p0):
    q = ternary(synth.rng_for(700, n, int(p0 * 100)), n, p0) if n else np.zeros(0, np.int8)
    bitmap, signs = oracle.bitcos_pack_flat(q)
    np.testing.assert_array_equal(bitmap, np.packbits(q != 0, bitorder="little"))
    np.testing.assert_array_equal(signs, np.packbits(q[q != 0] < 0, bitorder="little"))
    np.testing.assert_array_equal(oracle.bitcos_unpack_flat(bitmap, signs, n), q)


def test_hand_example():
    # presence 1,0,1,1,0,0,1,0,1 -> bytes 0x4D, 0x01; signs of the five
    # non-zeros (+,-,-,+,-) -> 0b10110
    q = np.array([1, 0, -1, -1, 0, 0, 1, 0, -1], np.int8)
    bitmap, signs = oracle.bitcos_pack_flat(q)
    assert bitmap.tolist() == [0x4D, 0x01] and signs.tolist() == [0x16]


def test_rejects_non_ternary():
    with pytest.raises(oracle.OracleReject):
        oracle.bitcos_pack_flat(np.array([0, 2, 1], np.int8))
    with pytest.raises(oracle.OracleReject):
        oracle.bitcos_pack_blocked(np.array([[0, -2, 1]], np.int8))


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "bitcos_sizes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                name, n, zpct, mb2, mbb, bits = line.split()
                rows.append((name, int(n), float(zpct), float(mb2), float(mbb), float(bits)))
    return rows


@pytest.mark.parametrize("row", _golden_rows(), ids=lambda r: r[0])
def test_page_sizes(row):
    """A vector with the page's weight count and zero share packs to the
    printed sizes: 2-bit n/4 bytes, BITCOS ceil(n/8) + ceil(nnz/8) bytes and
    2 - z bits per weight."""
    name, n, zpct, mb2, mbb, bits = row
    nnz = int(round(n * (1 - zpct / 100)))
    q = np.zeros(n, np.int8)
    idx = synth.rng_for(701, n).choice(n, nnz, replace=False)
    q[idx] = np.where(synth.rng_for(702, n).random(nnz) < 0.5, 1, -1)
    bitmap, signs = oracle.bitcos_pack_flat(q)
    total = bitmap.size + signs.size
    assert round(total / 1e6, 3) == mbb
    assert round(8 * total / n, 4) == bits
    assert round(oracle.payload_bytes(1, n) / 1e6, 3) == mb2   # one row of 2-bit planes


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 63), (5, 64), (7, 65), (16, 200), (9, 2560)])
def test_blocked_rows_are_flat_rows(rows, cols):
    w = synth.ternary(synth.rng_for(703, rows, cols), rows, cols, 0.42)
    bitmap, sign_off, signs = oracle.bitcos_pack_blocked(w)
    B = (cols + 63) // 64
    assert bitmap.shape == (rows, B) and sign_off[0] == 0
    assert (signs[-2:] == 0).all()
    for r in range(rows):
        flat_b, flat_s = oracle.bitcos_pack_flat(w[r])
        bits = np.unpackbits(bitmap[r].view(np.uint8), bitorder="little")
        np.testing.assert_array_equal(bits[:cols], np.unpackbits(flat_b, bitorder="little")[:cols])
        assert not bits[cols:].any()
        nnz = int((w[r] != 0).sum())
        assert sign_off[r + 1] - sign_off[r] == (nnz + 31) // 32
        sb = np.unpackbits(signs[sign_off[r]:sign_off[r + 1]].view(np.uint8), bitorder="little")
        np.testing.assert_array_equal(sb[:nnz], np.unpackbits(flat_s, bitorder="little")[:nnz])
        assert not sb[nnz:].any()


@pytest.mark.parametrize("rows,cols", [(1, 1), (4, 63), (33, 64), (17, 130), (64, 2560), (8, 6913)])
def test_bitcos_gemv_matches_plane_oracle(rows, cols):
    rng = synth.rng_for(704, rows, cols)
    w = synth.ternary(rng, rows, cols, float(rng.uniform(0.3, 0.6)))
    x = rng.integers(-128, 128, size=(1, ((cols + 63) // 64) * 64)).astype(np.int8)
    x[0, : min(cols, 5)] = -128
    xs = np.float32(rng.random() + 0.1)
    ws = float(synth.w_scale(w))
    y, yf = oracle.bitcos_gemv(*oracle.bitcos_pack_blocked(w), cols, ws, x[0], float(xs))
    ry, rf, err = oracle.gemm(oracle.pack(w), ws, x, np.array([xs], np.float32), cols)
    assert not err.any()
    np.testing.assert_array_equal(y, ry[0])
    np.testing.assert_array_equal(yf.view(np.uint32), rf[0].view(np.uint32))
    sel = np.array([rows - 1, 0])
    ys, _ = oracle.bitcos_gemv(*oracle.bitcos_pack_blocked(w), cols, ws, x[0], float(xs), rows=sel)
    np.testing.assert_array_equal(ys, ry[0][sel])

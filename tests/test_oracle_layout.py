"""Pins for the oracle's packer, unpacker and validator.

Each test checks the oracle against something the pages or plain mathematics
fix, not against a retyped copy of its own code:
  - the page's printed example file ("The .trit format, version 1" -- 3);
  - numpy's little-endian u64 view for bit order;
  - the page's 64-bit tail-mask formula for P2 (the oracle tests column
    indices instead);
  - size totals printed on the pages.
"""
import os

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_hex(name):
    data = bytearray()
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            parts = line.split()
            off = int(parts[0], 16)
            assert off == len(data)
            data += bytes(int(p, 16) for p in parts[1:])
    return bytes(data)


def _u64(b):
    return int(np.frombuffer(bytes(b), dtype="<u8")[0])


def test_worked_example_payload(orc):
    """W = [[+1,-1,0],[0,+1,+1]] packs to the page's 32 payload bytes."""
    blob = _read_hex("trit_v1_example.hex")
    assert blob[:4] == b"TRIT"
    payload_start = 0x80
    assert payload_start % 64 == 0
    w = np.array([[1, -1, 0], [0, 1, 1]], dtype=np.int8)
    got = orc.pack(w)
    assert got.shape == (2, 1, 16)
    assert got.tobytes() == blob[payload_start:payload_start + 32]
    # and the page's own bytes decode back, with the padding clear
    back = np.frombuffer(blob[payload_start:payload_start + 32], dtype=np.uint8).reshape(2, 1, 16)
    assert orc.verify(back, 3) == (0, -1)
    np.testing.assert_array_equal(orc.unpack(back, 3), w)


@pytest.mark.parametrize("cols", [1, 63, 64, 65, 200])
def test_bit_k_is_kth_lsb_of_little_endian_u64(orc, cols):
    for c in sorted({0, 7, 8, 31, 32, 63, 64, cols - 1} & set(range(cols))):
        for v, plane in ((1, 0), (-1, 1)):
            w = np.zeros((1, cols), dtype=np.int8)
            w[0, c] = v
            beats = orc.pack(w)[0]
            for b in range(beats.shape[0]):
                pos, neg = _u64(beats[b, :8]), _u64(beats[b, 8:])
                want = (1 << (c % 64)) if b == c // 64 else 0
                assert (pos, neg) == ((want, 0) if plane == 0 else (0, want))


ROWS = [1, 16, 17, 640]
COLS = [1, 3, 33, 63, 64, 65, 127, 128, 2560, 6912]


@pytest.mark.parametrize("rows", ROWS)
@pytest.mark.parametrize("cols", COLS)
def test_round_trip_and_padding(orc, rows, cols):
    rng = synth.rng_for(900, rows, cols)
    for w in (np.zeros((rows, cols), np.int8), synth.ternary(rng, rows, cols, 0.42)):
        p = orc.pack(w)
        assert p.shape == (rows, (cols + 63) // 64, 16)
        assert orc.verify(p, cols) == (0, -1)
        np.testing.assert_array_equal(orc.unpack(p, cols), w)


def test_two_bits_per_weight_and_byte_len(orc):
    for rows, cols in [(2560, 2560), (640, 2560), (6912, 2560), (2560, 6912), (3, 64), (1, 128)]:
        nbytes = orc.payload_bytes(rows, cols)
        assert nbytes * 8 == 2 * rows * cols  # exactly 2.000 bits per weight when cols % 64 == 0
    # ragged column counts pay for whole beats
    assert orc.payload_bytes(16, 33) == 16 * 16
    assert orc.payload_bytes(1, 65) == 32


def _golden_numbers():
    out = {}
    with open(os.path.join(GOLDEN, "bitnet_shapes.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                out[k] = int(v)
    return out


def test_stack_totals(orc):
    g = _golden_numbers()
    items = list(synth.stack_items())
    assert len(items) == g["tensors"]
    trits = sum(N * K for _, _, _, N, K in items)
    assert trits == g["total_trits"]
    assert sum(orc.payload_bytes(N, K) for _, _, _, N, K in items) * 4 == trits
    sizes = {name: N * K for name, N, K in synth.PROJECTIONS}
    assert sizes["q"] == g["q_proj_weights"] and sizes["up"] == g["up_proj_weights"]
    # the page's 2-bit sizes of those tensors (1.638 MB, 4.424 MB)
    assert round(orc.payload_bytes(2560, 2560) / 1e6, 3) == 1.638
    assert round(orc.payload_bytes(6912, 2560) / 1e6, 3) == 4.424


def test_pack_rejects_non_ternary(orc):
    w = np.zeros((3, 70), np.int8)
    w[2, 66] = 2
    with pytest.raises(orc.OracleReject) as e:
        orc.pack(w)
    assert e.value.code == orc.NOT_TERNARY and e.value.where == 2 * 70 + 66
    w[2, 66] = -128
    with pytest.raises(orc.OracleReject):
        orc.pack(w)


@pytest.mark.parametrize("k", [0, 31, 32, 63])
def test_verify_finds_both_set(orc, k):
    rows, cols = 5, 200
    p = orc.pack(synth.ternary(synth.rng_for(901, k), rows, cols, 0.4))
    B = p.shape[1]
    r, b = 3, 2
    if b * 64 + k >= cols:
        b = 1
    p[r, b, k // 8] |= 1 << (k % 8)
    p[r, b, 8 + k // 8] |= 1 << (k % 8)
    kinds, first = orc.verify(p, cols)
    assert kinds == orc.P1
    assert first == (r * B + b) * 64 + k
    with pytest.raises(orc.OracleReject) as e:
        orc.unpack(p, cols)
    assert e.value.code == orc.P1 and e.value.where == first


def _tail_mask(cols):
    """The page's tail mask, evaluated with Python's unbounded ints."""
    r = cols % 64
    return (1 << 64) - 1 if r == 0 else (1 << r) - 1


@pytest.mark.parametrize("rem", [1, 31, 32, 33, 63, 0])
def test_verify_padding_against_tail_mask(orc, rem):
    cols = 128 + rem
    B = (cols + 63) // 64
    for k in range(64):
        for plane in (0, 8):
            p = np.zeros((2, B, 16), np.uint8)
            p[1, B - 1, plane + k // 8] |= 1 << (k % 8)
            pos = _u64(p[1, B - 1, :8])
            neg = _u64(p[1, B - 1, 8:])
            dirty = ((pos | neg) & ~_tail_mask(cols) & ((1 << 64) - 1)) != 0
            kinds, first = orc.verify(p, cols)
            assert kinds == (orc.P2 if dirty else 0), (rem, k)
            assert first == ((1 * B + B - 1) * 64 + k if dirty else -1)


def test_verify_reports_first_violation(orc):
    cols = 100
    p = orc.pack(np.zeros((4, cols), np.int8))
    B = p.shape[1]
    p[3, 0, 0] = 1
    p[3, 0, 8] = 1          # P1 at row 3, beat 0, bit 0
    p[1, 1, 7] = 0x80       # P2 at row 1, beat 1, bit 63 (column 127 >= 100)
    kinds, first = orc.verify(p, cols)
    assert kinds == orc.P1 | orc.P2
    assert first == (1 * B + 1) * 64 + 63

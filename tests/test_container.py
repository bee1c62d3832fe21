"""The .trit v1 container ("The .trit format, version 1" -- 2, 3, 4).

Part 1 pins the oracle parser (oracle/container.py) to things other than
itself: the page's worked example (section 3), published FNV-1a-64 test
vectors, one planted violation per check of section 4, the truncation suite
the page describes (every prefix of the example's header region), and the
64-bit padding rule of 2.3.

Part 2 runs the library's C reader (include/trit_file.h; host code, no GPU)
on the same bytes and on seeded random files and corruptions, and requires it
to report exactly what the oracle reports.  The file writer below builds test
inputs with struct; it is neither the oracle nor the library."""
import os
import struct

import numpy as np
import pytest

from oracle import container as C

HERE = os.path.dirname(os.path.abspath(__file__))


def example_bytes() -> bytes:
    out = bytearray()
    for line in open(os.path.join(HERE, "golden", "trit_v1_example.hex")):
        if line.startswith("#") or not line.strip():
            continue
        out += bytes(int(x, 16) for x in line.split()[1:17])
    return bytes(out)


EX = example_bytes()


def patch(data: bytes, at: int, new: bytes) -> bytes:
    b = bytearray(data)
    b[at:at + len(new)] = new
    return bytes(b)


def write_file(tensors, config=b'{"hidden_size":3}', version=1, flags=0, hash_mode="fnv",
               pad_extra=0):
    """tensors: list of dicts name, dtype, dims, scale, payload(bytes), [offset], [flags],
    [reserved]; payload offsets are assigned in order (64-byte aligned) unless given."""
    recs = b""
    payload = bytearray()
    for t in tensors:
        if "offset" in t:
            off = t["offset"]
        else:
            off = (len(payload) + 63) // 64 * 64
        if len(payload) < off + len(t["payload"]):
            payload += b"\0" * (off + len(t["payload"]) - len(payload))
        payload[off:off + len(t["payload"])] = t["payload"]
        name = t["name"].encode() if isinstance(t["name"], str) else t["name"]
        r0, r1 = t.get("reserved", (0, 0))
        recs += struct.pack("<H", len(name)) + name
        recs += struct.pack("<BBBB", t["dtype"], len(t["dims"]), r0, r1)
        recs += struct.pack("<%dI" % len(t["dims"]), *t["dims"])
        recs += struct.pack("<fIQQ", t["scale"], t.get("flags", 0), off,
                            t.get("byte_len", len(t["payload"])))
    h = {"fnv": C.fnv1a64(bytes(payload)), "zero": 0}[hash_mode] if isinstance(hash_mode, str) \
        else hash_mode
    head = b"TRIT" + struct.pack("<IIQI", version, flags, h, len(config)) + config
    head += struct.pack("<I", len(tensors)) + recs
    head += b"\0" * ((-len(head)) % 64 + pad_extra)
    return head + bytes(payload)


def trit_payload(W: np.ndarray) -> bytes:
    """Planes of a small ternary matrix, bit by bit as 2.3 describes."""
    rows, cols = W.shape
    bpr = (cols + 63) // 64
    out = bytearray()
    for r in range(rows):
        for b in range(bpr):
            pos = neg = 0
            for k in range(64):
                c = 64 * b + k
                if c < cols and W[r, c] == 1:
                    pos |= 1 << k
                if c < cols and W[r, c] == -1:
                    neg |= 1 << k
            out += pos.to_bytes(8, "little") + neg.to_bytes(8, "little")
    return bytes(out)


# ---- part 1: the oracle against the page and the mathematics -----------------

def test_fnv1a64_published_vectors():
    assert C.fnv1a64(b"") == 0xCBF29CE484222325
    assert C.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert C.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_worked_example_fields():
    info = C.parse(EX)
    assert len(EX) == 160 and info["payload_start"] == 0x80 and info["payload_len"] == 32
    assert info["version"] == 1 and info["config"] == b'{"hidden_size":3}'
    assert info["payload_hash"] == 0x4A4ABD58B2E9F860
    (t,) = info["tensors"]
    assert (t["name"], t["dtype"], t["dims"], t["scale"], t["offset"], t["byte_len"]) == \
        ("w", C.DTYPE_TRIT, [2, 3], 0.5, 0, 32)
    np.testing.assert_array_equal(C.trit_matrix(EX, info, "w"), [[1, -1, 0], [0, 1, 1]])


def test_worked_example_hash_reading():
    """Checks 1-18 pass; the stored hash is not the standard FNV-1a-64 of the
    payload (check 19 fails) -- it is reproduced by the prime 2^44 + 0x1b3."""
    check, _ = C.first_violation(EX)
    assert check == 19
    assert C.fnv1a64(EX[0x80:], prime=(1 << 44) + 0x1B3) == 0x4A4ABD58B2E9F860
    assert C.first_violation(patch(EX, 12, struct.pack("<Q", C.fnv1a64(EX[0x80:]))))[0] == 0
    assert C.first_violation(patch(EX, 12, b"\0" * 8))[0] == 0      # 0 = absent, not checked


# offsets in the example: 0 magic, 4 version, 8 flags, 12 hash, 20 config_len,
# 24 config (17 B), 41 tensor_count, 45 name_len, 47 name, 48 dtype, 49 ndim,
# 50/51 reserved, 52 dims (2 x u32), 60 scale, 64 flags, 68 offset, 76 byte_len
PLANTED = [
    (1, patch(EX, 0, b"TRIX")),
    (2, patch(EX, 4, struct.pack("<I", 0))),
    (3, patch(EX, 4, struct.pack("<I", 2))),
    (4, patch(EX, 8, struct.pack("<I", 1))),
    (5, EX[:50]),
    (6, patch(EX, 20, struct.pack("<I", 16 * 1024 * 1024 + 1))),
    (6, patch(EX, 25, b"\xff")),
    (7, patch(EX, 45, struct.pack("<H", 0))),
    (7, patch(EX, 47, b"\xc3")),
    (8, patch(EX, 48, b"\x03")),
    (8, patch(EX, 49, b"\x00")),
    (8, patch(EX, 49, b"\x05")),
    (8, patch(EX, 50, b"\x01")),
    (8, patch(EX, 51, b"\x01")),
    (8, patch(EX, 64, struct.pack("<I", 4))),
    (8, patch(EX, 41, struct.pack("<I", 1048577))),
    (10, patch(EX, 60, struct.pack("<f", 0.0))),
    (10, patch(EX, 60, struct.pack("<f", -0.5))),
    (10, patch(EX, 60, struct.pack("<f", float("nan")))),
    (10, patch(EX, 60, struct.pack("<f", float("inf")))),
    (11, patch(EX, 68, struct.pack("<Q", 32))),
    (12, patch(EX, 76, struct.pack("<Q", 48))),
    (12, patch(EX, 68, struct.pack("<Q", 64))),
    (14, write_file([dict(name="w", dtype=1, dims=[6], scale=0.5, payload=EX[0x80:])])),
    (15, patch(EX, 52, struct.pack("<I", 1))),
    (16, patch(EX, 48, b"\x00")),
    (17, patch(EX, 0x80 + 8, b"\x03")),
    (18, patch(EX, 0x80, b"\x09")),
    (18, patch(EX, 0x90 + 8, b"\x00\x00\x00\x00\x00\x00\x00\x80")),
]


@pytest.mark.parametrize("check,data", PLANTED, ids=[f"{c}-{i}" for i, (c, _) in enumerate(PLANTED)])
def test_oracle_reports_each_planted_violation(check, data):
    got, msg = C.first_violation(data)
    assert got == check, msg


def test_check9_shape_overflow():
    f = write_file([dict(name="a", dtype=0, dims=[2**32 - 1] * 3, scale=1.0, payload=b"",
                         byte_len=0)])
    assert C.first_violation(f)[0] == 9
    f = write_file([dict(name="a", dtype=0, dims=[2**32 - 1, 2**32 - 1], scale=1.0, payload=b"",
                         byte_len=0)])
    assert C.first_violation(f)[0] == 16       # fits 64 bits; byte_len 0 is wrong


def test_check7_duplicates_and_check13_overlap():
    w = trit_payload(np.array([[1, 0, -1]]))
    a = dict(name="a", dtype=1, dims=[1, 3], scale=1.0, payload=w)
    assert C.first_violation(write_file([a, dict(a)]))[0] == 7
    b = dict(name="b", dtype=1, dims=[1, 3], scale=1.0, payload=w, offset=0)
    assert C.first_violation(write_file([a, b]))[0] == 13
    e = dict(name="e", dtype=0, dims=[0], scale=1.0, payload=b"", offset=0)   # empty extent
    assert C.first_violation(write_file([a, e]))[0] == 0


def test_truncation_suite():
    """Every prefix of the example that cuts the header region is rejected as
    truncated; cutting the payload leaves the tensor's extent past the end."""
    for n in range(0, 0x80):
        assert C.first_violation(EX[:n])[0] == 5, n
    for n in range(0x80, len(EX)):
        assert C.first_violation(EX[:n])[0] == 12, n


@pytest.mark.parametrize("cols", [1, 31, 32, 33, 63, 64, 65, 127])
def test_p2_tail_mask_is_64_bit(cols):
    W = np.zeros((2, cols), np.int8)
    W[1, cols - 1] = -1
    pay = bytearray(trit_payload(W))
    f = write_file([dict(name="w", dtype=1, dims=[2, cols], scale=1.0, payload=bytes(pay))])
    assert C.first_violation(f)[0] == 0
    bpr = (cols + 63) // 64
    if cols % 64:
        k = cols % 64                       # first padding bit of the last beat
        last = (1 * bpr + bpr - 1) * 16
        pos = int.from_bytes(pay[last:last + 8], "little") | (1 << k)
        pay[last:last + 8] = pos.to_bytes(8, "little")
        f = write_file([dict(name="w", dtype=1, dims=[2, cols], scale=1.0, payload=bytes(pay))])
        assert C.first_violation(f)[0] == 18


def test_p1_names_row_beat_column():
    W = np.zeros((3, 130), np.int8)
    pay = bytearray(trit_payload(W))
    o = (2 * 3 + 1) * 16                    # row 2, beat 1
    pay[o:o + 8] = (1 << 5).to_bytes(8, "little")
    pay[o + 8:o + 16] = (1 << 5).to_bytes(8, "little")
    f = write_file([dict(name="t", dtype=1, dims=[3, 130], scale=1.0, payload=bytes(pay))])
    check, msg = C.first_violation(f)
    assert check == 17 and "row 2 beat 1 col 69" in msg


# ---- part 2: the library's reader against the oracle ------------------------

@pytest.fixture(scope="module")
def tf():
    from bit_plane_select_gb300 import build
    build.build()
    from bit_plane_select_gb300 import trit_file
    return trit_file


def lib_check(tf, data: bytes) -> int:
    try:
        f = tf.TritFile.open_memory(data)
    except tf.TritFileError as e:
        return e.status
    try:
        f.verify()
    except tf.TritFileError as e:
        return e.status
    finally:
        f.close()
    return 0


def test_library_fnv_matches(tf):
    rng = np.random.default_rng(7)
    for n in (0, 1, 7, 64, 1000):
        d = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        assert tf.trit_fnv1a64(d) == C.fnv1a64(d)


def test_library_reads_the_worked_example(tf):
    f = tf.TritFile.open_memory(EX)
    assert len(f) == 1 and f.payload_start == 0x80 and f.payload_hash == 0x4A4ABD58B2E9F860
    assert f.config == b'{"hidden_size":3}'
    t = f.tensor(0)
    assert (t["name"], t["dtype"], t["dims"], t["scale"], t["offset"], t["byte_len"]) == \
        ("w", 1, [2, 3], 0.5, 0, 32)
    assert t["bytes"] == EX[0x80:]
    assert f.find("w") == 0 and f.find("x") == -1
    with pytest.raises(tf.TritFileError) as e:
        f.verify()
    assert e.value.status == 19
    f.close()


@pytest.mark.parametrize("check,data", PLANTED, ids=[f"{c}-{i}" for i, (c, _) in enumerate(PLANTED)])
def test_library_agrees_on_planted_violations(tf, check, data):
    assert lib_check(tf, data) == check


def test_library_truncation_suite(tf):
    for n in range(0, len(EX)):
        assert lib_check(tf, EX[:n]) == C.first_violation(EX[:n])[0], n


def random_file(rng) -> bytes:
    tensors = []
    for i in range(int(rng.integers(1, 6))):
        kind = int(rng.integers(0, 3))
        if kind == 1:
            rows, cols = int(rng.integers(1, 6)), int(rng.integers(1, 200))
            W = rng.integers(-1, 2, size=(rows, cols)).astype(np.int8)
            tensors.append(dict(name=f"t{i:02d}.w", dtype=1, dims=[rows, cols],
                                scale=float(rng.uniform(0.1, 2)), payload=trit_payload(W)))
        else:
            dims = [int(d) for d in rng.integers(1, 5, size=int(rng.integers(1, 5)))]
            n = int(np.prod(dims)) * (4 if kind == 0 else 2)
            tensors.append(dict(name=f"t{i:02d}.d", dtype=kind, dims=dims, scale=1.0,
                                payload=rng.integers(0, 256, n, dtype=np.uint8).tobytes()))
    return write_file(tensors, config=b'{"k":' + str(int(rng.integers(0, 99))).encode() + b"}",
                      hash_mode="fnv" if rng.random() < 0.7 else "zero")


def test_library_matches_oracle_on_random_files_and_corruptions(tf):
    rng = np.random.default_rng(20260)
    for trial in range(60):
        data = random_file(rng)
        info = C.parse(data)
        f = tf.TritFile.open_memory(data)
        assert len(f) == len(info["tensors"]) and f.payload_start == info["payload_start"]
        for i, t in enumerate(info["tensors"]):
            g = f.tensor(i)
            assert (g["name"], g["dtype"], g["dims"], g["offset"], g["byte_len"]) == \
                (t["name"], t["dtype"], t["dims"], t["offset"], t["byte_len"])
            assert np.float32(g["scale"]) == np.float32(t["scale"])
            assert g["bytes"] == C.tensor_bytes(data, info, t["name"])
            assert f.find(t["name"]) == i
        f.close()
        assert lib_check(tf, data) == C.first_violation(data)[0] == 0
        # corruptions: one byte of the header region, or one payload byte
        for _ in range(20):
            b = bytearray(data)
            at = int(rng.integers(0, info["payload_start"] if rng.random() < 0.8 else len(b)))
            b[at] = int(rng.integers(0, 256))
            assert lib_check(tf, bytes(b)) == C.first_violation(bytes(b))[0], (trial, at)


def test_open_from_path(tf, tmp_path):
    p = tmp_path / "example.trit"
    p.write_bytes(EX)
    with tf.TritFile.open(str(p)) as f:
        assert f.tensor(0)["bytes"] == EX[0x80:]
    empty = tmp_path / "empty.trit"
    empty.write_bytes(b"")
    with pytest.raises(tf.TritFileError) as e:
        tf.TritFile.open(str(empty))
    assert e.value.status == 5
    with pytest.raises(tf.TritFileError) as e:
        tf.TritFile.open(str(tmp_path / "missing.trit"))
    assert e.value.status == 32

"""CPU oracle for the .trit v1 container: a plain parser and validator.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``.  It shares no code with the
library's C reader (``bit_plane_select_gb300/csrc/trit_file.cpp``); the tests
run both on the same bytes and compare what they report.

Follows "The .trit format, version 1":
  - 2 File layout (header fields, little-endian, payload_start a multiple of 64),
  - 2.1 Header fields, 2.2 Tensor record, 2.3 Ternary payload, 2.4 Dense payload,
  - 4 Validation: checks 1-16 at open, 17-19 on request, each reported with the
    number the page gives it.

Readings where the page is silent (the C reader takes the same ones):
  - a read past the end of the data -- including a file shorter than the
    magic -- is check 5 (truncated);
  - tensor_count above 1,048,576 (a bound the layout table states but the
    check list does not number) is reported as check 8 (a record field out of
    range);
  - a tensor name that is not valid UTF-8 is check 7 (name);
  - the zero padding before payload_start is located, not inspected; a file
    that ends before payload_start is check 5;
  - order of the checks: the header fields as they are read (1, 2/3, 4, 6,
    then the tensor count); each record as it is read -- name length and UTF-8
    (7), ndim (8) before the dims are read, then after the whole record dtype,
    reserved bytes and flags (8), shape product (9), scale (10), offset
    alignment (11); once the last record is read payload_start is known and
    each record in file order gets 12, 14, 15/16; then duplicate names (7),
    then overlapping extents (13).  Extents of zero bytes overlap nothing; a
    size product that does not fit 64 bits never equals byte_len;
  - verification scans ternary tensors in record order, rows in order; within
    a row every beat's P1 (17) before the row's P2 (18); then the hash (19),
    skipped when the stored hash is 0;
  - the hash is the standard FNV-1a-64 (offset basis 0xcbf29ce484222325,
    prime 0x100000001b3), as section 2 names it.  The page's own example in
    section 3 stores a value that this does not reproduce (the prime
    0x1000000001b3 does); the example therefore fails check 19 and passes the
    others.
"""
from __future__ import annotations

import math
import struct

import numpy as np

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MAX_CONFIG = 16 * 1024 * 1024
MAX_TENSORS = 1048576
DTYPE_F32, DTYPE_TRIT, DTYPE_BF16 = 0, 1, 2
ELEM = {DTYPE_F32: 4, DTYPE_BF16: 2}


class ContainerError(Exception):
    """A rejected file: `check` is the number of the failed check (1-19)."""

    def __init__(self, check: int, what: str = ""):
        super().__init__(f"check {check}: {what}")
        self.check = check


def fnv1a64(data: bytes, prime: int = FNV_PRIME, basis: int = FNV_OFFSET) -> int:
    """FNV-1a, 64-bit: for each byte, xor it in, then multiply by the prime mod 2^64."""
    h = basis
    for b in data:
        h ^= b
        h = (h * prime) & 0xFFFFFFFFFFFFFFFF
    return h


class _Reader:
    def __init__(self, data: bytes):
        self.data = data
        self.pos = 0

    def take(self, n: int) -> bytes:
        if self.pos + n > len(self.data):
            raise ContainerError(5, "truncated")
        b = self.data[self.pos:self.pos + n]
        self.pos += n
        return b

    def u8(self):
        return self.take(1)[0]

    def u16(self):
        return struct.unpack("<H", self.take(2))[0]

    def u32(self):
        return struct.unpack("<I", self.take(4))[0]

    def u64(self):
        return struct.unpack("<Q", self.take(8))[0]

    def f32(self):
        return struct.unpack("<f", self.take(4))[0]


def beats_per_row(cols: int) -> int:
    return (cols + 63) // 64


def parse(data: bytes) -> dict:
    """Checks 1-16.  Returns the header fields, the records and payload_start."""
    r = _Reader(bytes(data))
    if r.take(4) != b"TRIT":
        raise ContainerError(1, "magic")
    version = r.u32()
    if version == 0:
        raise ContainerError(2, "version 0")
    if version > 1:
        raise ContainerError(3, f"version {version}")
    flags = r.u32()
    if flags != 0:
        raise ContainerError(4, f"header flags {flags:#x}")
    payload_hash = r.u64()
    config_len = r.u32()
    if config_len > MAX_CONFIG:
        raise ContainerError(6, "config_len")
    config = r.take(config_len)
    try:
        config.decode("utf-8")
    except UnicodeDecodeError:
        raise ContainerError(6, "config not UTF-8")
    count = r.u32()
    if count > MAX_TENSORS:
        raise ContainerError(8, "tensor_count")
    tensors = []
    for _ in range(count):
        name_len = r.u16()
        if name_len == 0 or name_len > 1024:
            raise ContainerError(7, "name_len")
        name_b = r.take(name_len)
        try:
            name = name_b.decode("utf-8")
        except UnicodeDecodeError:
            raise ContainerError(7, "name not UTF-8")
        dtype, ndim, res0, res1 = r.u8(), r.u8(), r.u8(), r.u8()
        if not 1 <= ndim <= 4:
            raise ContainerError(8, "ndim")
        dims = [r.u32() for _ in range(ndim)]
        scale = r.f32()
        tflags = r.u32()
        offset = r.u64()
        byte_len = r.u64()
        if dtype not in (DTYPE_F32, DTYPE_TRIT, DTYPE_BF16) or res0 or res1 or tflags:
            raise ContainerError(8, "dtype / reserved / flags")
        prod = math.prod(dims)
        if prod >= 1 << 64:
            raise ContainerError(9, "shape product")
        if not math.isfinite(scale) or not scale > 0:
            raise ContainerError(10, "scale")
        if offset % 64:
            raise ContainerError(11, "offset alignment")
        tensors.append(dict(name=name, name_bytes=name_b, dtype=dtype, dims=dims, scale=scale,
                            offset=offset, byte_len=byte_len, prod=prod))
    end_records = r.pos
    payload_start = (end_records + 63) // 64 * 64
    if payload_start > len(r.data):
        raise ContainerError(5, "truncated before payload")
    payload_len = len(r.data) - payload_start
    for t in tensors:
        if t["offset"] + t["byte_len"] > payload_len:
            raise ContainerError(12, f"extent of {t['name']}")
        if t["dtype"] == DTYPE_TRIT:
            if len(t["dims"]) != 2:
                raise ContainerError(14, f"{t['name']} not 2-D")
            rows, cols = t["dims"]
            if t["byte_len"] != rows * beats_per_row(cols) * 16:
                raise ContainerError(15, f"{t['name']} byte_len")
        else:
            if t["byte_len"] != t["prod"] * ELEM[t["dtype"]]:
                raise ContainerError(16, f"{t['name']} byte_len")
    names = [t["name_bytes"] for t in tensors]
    if len(set(names)) != len(names):
        raise ContainerError(7, "duplicate name")
    ext = sorted((t["offset"], t["offset"] + t["byte_len"]) for t in tensors if t["byte_len"] > 0)
    for (a0, a1), (b0, b1) in zip(ext, ext[1:]):
        if b0 < a1:
            raise ContainerError(13, "overlap")
    return dict(version=version, payload_hash=payload_hash, config=config, tensors=tensors,
                payload_start=payload_start, payload_len=payload_len)


def verify(data: bytes, info: dict | None = None) -> dict:
    """Checks 17-19 on a file that passed `parse`."""
    data = bytes(data)
    if info is None:
        info = parse(data)
    ps = info["payload_start"]
    for t in info["tensors"]:
        if t["dtype"] != DTYPE_TRIT:
            continue
        rows, cols = t["dims"]
        bpr = beats_per_row(cols)
        tail = 0xFFFFFFFFFFFFFFFF if cols % 64 == 0 else (1 << (cols % 64)) - 1
        base = ps + t["offset"]
        for row in range(rows):
            for b in range(bpr):
                o = base + (row * bpr + b) * 16
                pos = int.from_bytes(data[o:o + 8], "little")
                neg = int.from_bytes(data[o + 8:o + 16], "little")
                both = pos & neg
                if both:
                    k = (both & -both).bit_length() - 1
                    raise ContainerError(17, f"P1 {t['name']} row {row} beat {b} col {b * 64 + k}")
            o = base + (row * bpr + bpr - 1) * 16
            pos = int.from_bytes(data[o:o + 8], "little")
            neg = int.from_bytes(data[o + 8:o + 16], "little")
            if (pos | neg) & ~tail & 0xFFFFFFFFFFFFFFFF:
                raise ContainerError(18, f"P2 {t['name']} row {row}")
    if info["payload_hash"] != 0 and fnv1a64(data[ps:]) != info["payload_hash"]:
        raise ContainerError(19, "payload hash")
    return info


def first_violation(data: bytes) -> tuple[int, str]:
    """(0, "") for a file that opens and verifies, else (check, message)."""
    try:
        verify(data)
    except ContainerError as e:
        return e.check, str(e)
    return 0, ""


def tensor_bytes(data: bytes, info: dict, name: str) -> bytes:
    t = next(t for t in info["tensors"] if t["name"] == name)
    o = info["payload_start"] + t["offset"]
    return bytes(data)[o:o + t["byte_len"]]


def trit_matrix(data: bytes, info: dict, name: str) -> np.ndarray:
    """Decode a ternary tensor bit by bit (2.3): W[r][64b+k] = +1 if pos bit k,
    -1 if neg bit k, else 0."""
    t = next(t for t in info["tensors"] if t["name"] == name)
    rows, cols = t["dims"]
    bpr = beats_per_row(cols)
    raw = tensor_bytes(data, info, name)
    W = np.zeros((rows, cols), np.int8)
    for row in range(rows):
        for b in range(bpr):
            o = (row * bpr + b) * 16
            pos = int.from_bytes(raw[o:o + 8], "little")
            neg = int.from_bytes(raw[o + 8:o + 16], "little")
            for k in range(64):
                c = b * 64 + k
                if c >= cols:
                    break
                if (pos >> k) & 1:
                    W[row, c] = 1
                elif (neg >> k) & 1:
                    W[row, c] = -1
    return W

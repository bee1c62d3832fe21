"""Thin binding of the .trit v1 container reader declared in include/trit_file.h.

Every parse, check and copy happens in libtrit.so; this module marshals
arguments and raises TritFileError with the library's status (the number of
the failed check) and message.

    with TritFile.open(path) as f:        # checks 1-16
        f.verify()                        # checks 17-19 (host)
        planes = f.upload("w")            # a uint8 CUDA tensor [rows, beats, 16]
"""
from __future__ import annotations

import ctypes

import torch

from . import TritError, _check, _stream, lib

F32, TRIT, BF16 = 0, 1, 2


class TritFileError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"check {status}: {message}" if 1 <= status <= 19 else
                         f"status {status}: {message}")
        self.status = status


class TritTensorInfo(ctypes.Structure):
    _fields_ = [("name", ctypes.c_void_p), ("name_len", ctypes.c_uint32),
                ("dtype", ctypes.c_uint32), ("ndim", ctypes.c_uint32),
                ("dims", ctypes.c_uint32 * 4), ("scale", ctypes.c_float),
                ("reserved", ctypes.c_uint32), ("offset", ctypes.c_uint64),
                ("byte_len", ctypes.c_uint64), ("data", ctypes.c_void_p)]


_ready = False


def _lib():
    global _ready
    L = lib()
    if not _ready:
        p, u32, u64, sz = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t
        L.trit_file_open.argtypes = [ctypes.c_char_p, ctypes.POINTER(p), ctypes.c_char_p, sz]
        L.trit_file_open.restype = ctypes.c_int
        L.trit_file_open_memory.argtypes = [p, u64, ctypes.POINTER(p), ctypes.c_char_p, sz]
        L.trit_file_open_memory.restype = ctypes.c_int
        L.trit_file_close.argtypes = [p]
        L.trit_file_close.restype = None
        L.trit_file_verify.argtypes = [p, ctypes.c_char_p, sz]
        L.trit_file_verify.restype = ctypes.c_int
        L.trit_file_tensor_count.argtypes = [p]
        L.trit_file_tensor_count.restype = u32
        L.trit_file_tensor.argtypes = [p, u32, ctypes.POINTER(TritTensorInfo)]
        L.trit_file_tensor.restype = ctypes.c_int
        L.trit_file_find.argtypes = [p, ctypes.c_char_p, u32]
        L.trit_file_find.restype = ctypes.c_int64
        L.trit_file_config.argtypes = [p, ctypes.POINTER(u32)]
        L.trit_file_config.restype = p
        for n in ("trit_file_payload_hash", "trit_file_payload_start", "trit_file_payload_len"):
            getattr(L, n).argtypes = [p]
            getattr(L, n).restype = u64
        L.trit_fnv1a64.argtypes = [p, u64]
        L.trit_fnv1a64.restype = u64
        L.trit_file_upload.argtypes = [p, u32, p, p]
        L.trit_file_upload.restype = ctypes.c_int
        _ready = True
    return L


def trit_fnv1a64(data: bytes) -> int:
    buf = (ctypes.c_uint8 * len(data)).from_buffer_copy(data) if data else None
    return int(_lib().trit_fnv1a64(ctypes.cast(buf, ctypes.c_void_p) if buf else None, len(data)))


class TritFile:
    """An opened, header-validated .trit v1 file."""

    def __init__(self, handle, keep=None):
        self._h = handle
        self._keep = keep          # the caller's bytes for open_memory

    @classmethod
    def open(cls, path: str) -> "TritFile":
        h = ctypes.c_void_p()
        msg = ctypes.create_string_buffer(512)
        st = _lib().trit_file_open(path.encode(), ctypes.byref(h), msg, 512)
        if st != 0:
            raise TritFileError(st, msg.value.decode(errors="replace"))
        return cls(h)

    @classmethod
    def open_memory(cls, data: bytes) -> "TritFile":
        buf = (ctypes.c_uint8 * max(1, len(data))).from_buffer_copy(data or b"\0")
        h = ctypes.c_void_p()
        msg = ctypes.create_string_buffer(512)
        st = _lib().trit_file_open_memory(ctypes.cast(buf, ctypes.c_void_p), len(data),
                                          ctypes.byref(h), msg, 512)
        if st != 0:
            raise TritFileError(st, msg.value.decode(errors="replace"))
        return cls(h, buf)

    def close(self):
        if self._h:
            _lib().trit_file_close(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def verify(self):
        msg = ctypes.create_string_buffer(512)
        st = _lib().trit_file_verify(self._h, msg, 512)
        if st != 0:
            raise TritFileError(st, msg.value.decode(errors="replace"))

    def __len__(self):
        return int(_lib().trit_file_tensor_count(self._h))

    def tensor(self, i: int) -> dict:
        info = TritTensorInfo()
        st = _lib().trit_file_tensor(self._h, i, ctypes.byref(info))
        if st != 0:
            raise TritFileError(st, f"no tensor {i}")
        return dict(name=ctypes.string_at(info.name, info.name_len).decode(),
                    dtype=info.dtype, dims=list(info.dims[:info.ndim]), scale=info.scale,
                    offset=info.offset, byte_len=info.byte_len,
                    bytes=ctypes.string_at(info.data, info.byte_len) if info.byte_len else b"")

    def find(self, name: str) -> int:
        b = name.encode()
        return int(_lib().trit_file_find(self._h, b, len(b)))

    @property
    def config(self) -> bytes:
        n = ctypes.c_uint32()
        p = _lib().trit_file_config(self._h, ctypes.byref(n))
        return ctypes.string_at(p, n.value) if n.value else b""

    @property
    def payload_hash(self) -> int:
        return int(_lib().trit_file_payload_hash(self._h))

    @property
    def payload_start(self) -> int:
        return int(_lib().trit_file_payload_start(self._h))

    def upload(self, name_or_index, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """Copy a tensor's bytes unchanged into a CUDA tensor (uint8; ternary
        tensors shaped [rows, beats, 16], the layout trit_gemm reads)."""
        i = self.find(name_or_index) if isinstance(name_or_index, str) else int(name_or_index)
        if i < 0:
            raise KeyError(name_or_index)
        info = TritTensorInfo()
        if _lib().trit_file_tensor(self._h, i, ctypes.byref(info)) != 0:
            raise TritFileError(33, f"no tensor {i}")
        if out is None:
            shape = ((info.dims[0], (info.dims[1] + 63) // 64, 16) if info.dtype == TRIT
                     else (int(info.byte_len),))
            out = torch.empty(shape, dtype=torch.uint8, device="cuda")
        if out.numel() * out.element_size() < info.byte_len or not out.is_cuda:
            raise ValueError("out must be a CUDA tensor of at least byte_len bytes")
        _check(_lib().trit_file_upload(self._h, i, ctypes.c_void_p(out.data_ptr()),
                                       _stream(stream)), "trit_file_upload")
        return out


__all__ = ["TritFile", "TritFileError", "TritTensorInfo", "trit_fnv1a64", "F32", "TRIT", "BF16",
           "TritError"]

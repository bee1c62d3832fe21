"""bit_plane_select_gb300 -- ternary select-accumulate GEMV/GEMM over .trit v1
bit planes on GB300 (sm_103a).

This module is a thin ctypes binding of ``libtrit.so`` (declared in
``include/trit.h``): it checks tensor dtypes/devices and passes raw device
pointers and the current torch stream.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU fallback -- if the library is not
built, or the device is not an sm_103 GPU, the calls raise.

Functions carry the C names:
  trit_pack, trit_unpack, trit_verify, trit_quant_act, trit_quant_act_many,
  trit_gemv, trit_gemm, trit_gemm_many, trit_quant_gemv_many, trit_gemm_noalloc,
  trit_quant_act_folded, trit_intmlp_quant, trit_intmlp_gemv_many, trit_check_div127,
  trit_read_probe
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "TritError", "ERR_P1", "ERR_P2", "ERR_NOT_TERNARY", "ERR_NONFINITE", "ERR_TIMEOUT",
    "library_path", "lib", "payload_bytes", "k_pad", "trit_pack", "trit_unpack", "trit_verify",
    "trit_quant_act", "trit_quant_act_many", "trit_gemv", "trit_gemm", "trit_gemm_many",
    "trit_quant_gemv_many", "ProjList", "ActList", "QProjList", "TritProj", "TritAct",
    "TritQProj", "MAX_FUSED_K", "trit_gemm_noalloc", "NOALLOC_SCRATCH_BYTES",
    "trit_quant_act_folded", "trit_intmlp_quant", "trit_check_div127", "trit_read_probe",
    "trit_intmlp_gemv_many", "MlpProjList", "TritMlpProj", "PROBE_KINDS", "trit_issue_probe",
    "PLANES_READY", "TritMlpBlock", "MlpBlockList", "trit_mlp_tmax_bytes", "trit_mlp_gate_up",
    "trit_mlp_down",
]

ERR_P1 = 1
ERR_P2 = 2
ERR_NOT_TERNARY = 4
ERR_NONFINITE = 8
ERR_TIMEOUT = 16
MAX_FUSED_K = 73728
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024

_STATUS = {0: "TRIT_OK", 1: "TRIT_E_ARG", 2: "TRIT_E_SHAPE", 4: "TRIT_E_SCALE",
           6: "TRIT_E_CUDA", 7: "TRIT_E_DEVICE", 8: "TRIT_E_SCRATCH", 9: "TRIT_E_VALUE"}
BITCOS_MAX_K = 16384


class TritError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        super().__init__(f"{where}: {_STATUS.get(status, status)} {detail}".strip())
        self.status = status


class TritProj(ctypes.Structure):
    _fields_ = [("planes", ctypes.c_void_p), ("x_i8", ctypes.c_void_p),
                ("x_scale", ctypes.c_void_p), ("y_i32", ctypes.c_void_p),
                ("y_f32", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("w_scale", ctypes.c_float), ("flags", ctypes.c_uint32)]


class TritQProj(ctypes.Structure):
    _fields_ = [("planes", ctypes.c_void_p), ("x", ctypes.c_void_p), ("x_i8", ctypes.c_void_p),
                ("x_scale", ctypes.c_void_p), ("y_i32", ctypes.c_void_p),
                ("y_f32", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("w_scale", ctypes.c_float), ("flags", ctypes.c_uint32)]


class TritMlpProj(ctypes.Structure):
    _fields_ = [("planes", ctypes.c_void_p), ("a_gate", ctypes.c_void_p), ("a_up", ctypes.c_void_p),
                ("x_scale", ctypes.c_void_p), ("w_gate", ctypes.c_float), ("w_up", ctypes.c_float),
                ("h_i8", ctypes.c_void_p), ("h_scale", ctypes.c_void_p),
                ("y_i32", ctypes.c_void_p), ("y_f32", ctypes.c_void_p), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("w_scale", ctypes.c_float), ("reserved", ctypes.c_uint32)]


class TritMlpBlock(ctypes.Structure):
    _fields_ = [("gate_planes", ctypes.c_void_p), ("up_planes", ctypes.c_void_p),
                ("down_planes", ctypes.c_void_p), ("x", ctypes.c_void_p),
                ("x_scale", ctypes.c_void_p), ("a_gate", ctypes.c_void_p), ("a_up", ctypes.c_void_p),
                ("tmax", ctypes.c_void_p), ("h_i8", ctypes.c_void_p), ("h_scale", ctypes.c_void_p),
                ("y_i32", ctypes.c_void_p), ("y_f32", ctypes.c_void_p), ("K", ctypes.c_int64),
                ("F", ctypes.c_int64), ("N", ctypes.c_int64), ("w_gate", ctypes.c_float),
                ("w_up", ctypes.c_float), ("w_down", ctypes.c_float), ("flags", ctypes.c_uint32)]


class TritBitcosProj(ctypes.Structure):
    _fields_ = [("bitmap", ctypes.c_void_p), ("sign_off", ctypes.c_void_p), ("signs", ctypes.c_void_p),
                ("x_i8", ctypes.c_void_p), ("x_scale", ctypes.c_void_p), ("y_i32", ctypes.c_void_p),
                ("y_f32", ctypes.c_void_p), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("sign_words", ctypes.c_int64), ("w_scale", ctypes.c_float),
                ("reserved", ctypes.c_int32)]


class TritAct(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("x_i8", ctypes.c_void_p), ("x_scale", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("K", ctypes.c_int64)]


_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded libtrit.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with bit_plane_select_gb300.build.build() "
                "(needs nvcc); there is no fallback implementation")
        L = ctypes.CDLL(path)
        p, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        L.trit_status_string.restype = ctypes.c_char_p
        L.trit_status_string.argtypes = [ctypes.c_int]
        L.trit_last_cuda_error.restype = ctypes.c_char_p
        L.trit_last_cuda_error.argtypes = []
        L.trit_abi_version.restype = i32
        L.trit_payload_bytes.restype = i64
        L.trit_payload_bytes.argtypes = [i64, i64]
        L.trit_pack.argtypes = [p, i64, i64, f32, p, p, p, p]
        L.trit_unpack.argtypes = [p, i64, i64, p, p, p]
        L.trit_verify.argtypes = [p, i64, i64, p, p, p]
        L.trit_quant_act.argtypes = [p, i64, i64, p, p, p, p]
        L.trit_quant_act_many.argtypes = [p, i32, p, p]
        L.trit_gemv.argtypes = [p, f32, p, f32, i64, i64, p, p, p, p]
        L.trit_gemm.argtypes = [p, f32, p, p, i64, i64, i64, p, p, p, p]
        L.trit_gemm_many.argtypes = [p, i32, p, p]
        L.trit_quant_gemv_many.argtypes = [p, i32, p, p]
        L.trit_intmlp_gemv_many.argtypes = [p, i32, p, p]
        L.trit_mlp_tmax_bytes.restype = i64
        L.trit_mlp_tmax_bytes.argtypes = [i64]
        L.trit_mlp_gate_up.argtypes = [p, i32, p, p]
        L.trit_mlp_down.argtypes = [p, i32, p, p]
        L.trit_gemm_noalloc.argtypes = [p, f32, p, p, i64, i64, i64, p, p, p, p]
        L.trit_quant_act_folded.argtypes = [p, p, i64, i64, f32, p, p, p, p]
        L.trit_intmlp_quant.argtypes = [p, p, i64, i64, f32, f32, p, p, p, p]
        L.trit_check_div127.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
        L.trit_read_probe.argtypes = [p, i64, p, p]
        L.trit_issue_probe.argtypes = [i32, i32, i32, i64, p, p, p]
        L.trit_bitcos_pack.argtypes = [p, i64, i64, p, p, p, p]
        L.trit_bitcos_gemv_many.argtypes = [p, i32, p]
        for name in ("trit_pack", "trit_unpack", "trit_verify", "trit_quant_act",
                     "trit_quant_act_many", "trit_gemv", "trit_gemm", "trit_gemm_many",
                     "trit_quant_gemv_many", "trit_gemm_noalloc", "trit_quant_act_folded",
                     "trit_intmlp_quant", "trit_check_div127", "trit_read_probe",
                     "trit_intmlp_gemv_many", "trit_bitcos_pack", "trit_bitcos_gemv_many",
                     "trit_issue_probe", "trit_mlp_gate_up", "trit_mlp_down"):
            getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, where: str):
    if status != 0:
        detail = lib().trit_last_cuda_error().decode() if status == 6 else ""
        raise TritError(status, where, detail)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor | None, dtype, name: str, optional: bool = False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def payload_bytes(N: int, K: int) -> int:
    return int(lib().trit_payload_bytes(N, K))


def k_pad(K: int) -> int:
    """Row stride of the int8 activations: 64 * ceil(K / 64)."""
    return ((K + 63) // 64) * 64


def _err(err_flag, device):
    if err_flag is None:
        err_flag = torch.zeros(1, dtype=torch.int32, device=device)
    return err_flag


def trit_pack(w: torch.Tensor, w_scale: float, planes=None, scale_out=None, err_flag=None,
              stream=None):
    """int8 [N, K] ternary -> planes uint8 [N, ceil(K/64), 16].  Returns (planes, err_flag)."""
    N, K = w.shape
    if planes is None:
        planes = torch.empty((N, (K + 63) // 64, 16), dtype=torch.uint8, device=w.device)
    err_flag = _err(err_flag, w.device)
    _check(lib().trit_pack(_dev(w, torch.int8, "w"), N, K, float(w_scale),
                           _dev(planes, torch.uint8, "planes"),
                           _dev(scale_out, torch.float32, "scale_out", True),
                           _dev(err_flag, torch.int32, "err_flag"), _stream(stream)), "trit_pack")
    return planes, err_flag


def trit_unpack(planes: torch.Tensor, K: int, w=None, err_flag=None, stream=None):
    N = planes.shape[0]
    if w is None:
        w = torch.empty((N, K), dtype=torch.int8, device=planes.device)
    err_flag = _err(err_flag, planes.device)
    _check(lib().trit_unpack(_dev(planes, torch.uint8, "planes"), N, K, _dev(w, torch.int8, "w"),
                             _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_unpack")
    return w, err_flag


def trit_verify(planes: torch.Tensor, K: int, err_flag=None, first_bad=None, stream=None):
    """Returns (err_flag, first_bad); first_bad is an int64 tensor initialised to -1
    (UINT64_MAX) when not given."""
    N = planes.shape[0]
    err_flag = _err(err_flag, planes.device)
    if first_bad is None:
        first_bad = torch.full((1,), -1, dtype=torch.int64, device=planes.device)
    _check(lib().trit_verify(_dev(planes, torch.uint8, "planes"), N, K,
                             _dev(err_flag, torch.int32, "err_flag"),
                             _dev(first_bad, torch.int64, "first_bad"), _stream(stream)),
           "trit_verify")
    return err_flag, first_bad


def trit_quant_act(x: torch.Tensor, x_i8=None, x_scale=None, err_flag=None, stream=None):
    """fp32 [M, K] -> (x_i8 [M, K_pad], x_scale [M], err_flag)."""
    if x.dim() == 1:
        x = x.unsqueeze(0)
    M, K = x.shape
    if x_i8 is None:
        x_i8 = torch.empty((M, k_pad(K)), dtype=torch.int8, device=x.device)
    if x_scale is None:
        x_scale = torch.empty(M, dtype=torch.float32, device=x.device)
    err_flag = _err(err_flag, x.device)
    _check(lib().trit_quant_act(_dev(x, torch.float32, "x"), M, K, _dev(x_i8, torch.int8, "x_i8"),
                                _dev(x_scale, torch.float32, "x_scale"),
                                _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_quant_act")
    return x_i8, x_scale, err_flag


def trit_gemm(planes: torch.Tensor, w_scale: float, x_i8: torch.Tensor, x_scale: torch.Tensor,
              K: int, y_i32=None, y_f32=None, err_flag=None, stream=None, want=("i32", "f32")):
    """y = W x for M = x_i8.shape[0] rows.  Returns (y_i32, y_f32, err_flag)."""
    N = planes.shape[0]
    M = x_i8.shape[0] if x_i8.dim() == 2 else 1
    if y_i32 is None and "i32" in want:
        y_i32 = torch.empty((M, N), dtype=torch.int32, device=planes.device)
    if y_f32 is None and "f32" in want:
        y_f32 = torch.empty((M, N), dtype=torch.float32, device=planes.device)
    err_flag = _err(err_flag, planes.device)
    _check(lib().trit_gemm(_dev(planes, torch.uint8, "planes"), float(w_scale),
                           _dev(x_i8, torch.int8, "x_i8"), _dev(x_scale, torch.float32, "x_scale"),
                           M, N, K, _dev(y_i32, torch.int32, "y_i32", True),
                           _dev(y_f32, torch.float32, "y_f32", True),
                           _dev(err_flag, torch.int32, "err_flag"), _stream(stream)), "trit_gemm")
    return y_i32, y_f32, err_flag


def trit_gemm_noalloc(planes: torch.Tensor, w_scale: float, x_i8: torch.Tensor,
                      x_scale: torch.Tensor, K: int, y_i32, y_f32, err_flag, stream=None):
    """trit_gemm through the entry point that allocates nothing: every buffer,
    outputs and err_flag included, is the caller's (pass None for one output to
    skip it).  Returns (y_i32, y_f32, err_flag)."""
    N = planes.shape[0]
    M = x_i8.shape[0] if x_i8.dim() == 2 else 1
    _check(lib().trit_gemm_noalloc(_dev(planes, torch.uint8, "planes"), float(w_scale),
                                   _dev(x_i8, torch.int8, "x_i8"),
                                   _dev(x_scale, torch.float32, "x_scale"), M, N, K,
                                   _dev(y_i32, torch.int32, "y_i32", True),
                                   _dev(y_f32, torch.float32, "y_f32", True),
                                   _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_gemm_noalloc")
    return y_i32, y_f32, err_flag


def trit_quant_act_folded(x: torch.Tensor, gain: torch.Tensor, eps: float, x_i8=None,
                          x_scale=None, err_flag=None, stream=None):
    """Folded normalisation + quantisation: codes of x * gain, scale absmax / rms.
    fp32 [M, K] -> (x_i8 [M, K_pad], x_scale [M], err_flag)."""
    if x.dim() == 1:
        x = x.unsqueeze(0)
    M, K = x.shape
    if x_i8 is None:
        x_i8 = torch.empty((M, k_pad(K)), dtype=torch.int8, device=x.device)
    if x_scale is None:
        x_scale = torch.empty(M, dtype=torch.float32, device=x.device)
    err_flag = _err(err_flag, x.device)
    _check(lib().trit_quant_act_folded(_dev(x, torch.float32, "x"), _dev(gain, torch.float32, "gain"),
                                       M, K, float(eps), _dev(x_i8, torch.int8, "x_i8"),
                                       _dev(x_scale, torch.float32, "x_scale"),
                                       _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_quant_act_folded")
    return x_i8, x_scale, err_flag


def trit_intmlp_quant(a_gate: torch.Tensor, a_up: torch.Tensor, w_scale_gate: float,
                      w_scale_up: float, x_scale: torch.Tensor, h_i8=None, h_scale=None,
                      stream=None):
    """relu(a_gate)^2 * a_up kept integer, quantised for the next projection.
    int32 [M, N] x 2 -> (h_i8 [M, N_pad], h_scale [M])."""
    if a_gate.dim() == 1:
        a_gate, a_up = a_gate.unsqueeze(0), a_up.unsqueeze(0)
    M, N = a_gate.shape
    if h_i8 is None:
        h_i8 = torch.empty((M, k_pad(N)), dtype=torch.int8, device=a_gate.device)
    if h_scale is None:
        h_scale = torch.empty(M, dtype=torch.float32, device=a_gate.device)
    _check(lib().trit_intmlp_quant(_dev(a_gate, torch.int32, "a_gate"), _dev(a_up, torch.int32, "a_up"),
                                   M, N, float(w_scale_gate), float(w_scale_up),
                                   _dev(x_scale, torch.float32, "x_scale"),
                                   _dev(h_i8, torch.int8, "h_i8"),
                                   _dev(h_scale, torch.float32, "h_scale"), _stream(stream)),
           "trit_intmlp_quant")
    return h_i8, h_scale


def trit_read_probe(buf: torch.Tensor, sink: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Read every byte of the CUDA tensor `buf` once (a plain coalesced stream);
    the launch's duration measures the device's memory read rate."""
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    nbytes = buf.numel() * buf.element_size()
    if sink is None:
        sink = torch.zeros(1, dtype=torch.int32, device=buf.device)
    _check(lib().trit_read_probe(ctypes.c_void_p(buf.data_ptr()), nbytes - nbytes % 16,
                                 ctypes.c_void_p(sink.data_ptr()), _stream(stream)),
           "trit_read_probe")
    return sink


# instruction kinds of trit_issue_probe (TRIT_PROBE_* in include/trit.h)
PROBE_KINDS = {"dp4a": 0, "lop3": 1, "prmt": 2, "shf": 3, "imad": 4, "iadd": 5, "shfl": 6,
               "lds32": 7, "lds128": 8, "dp4a+lop3": 9,
               "dp4a.su": 10}


def trit_issue_probe(kind: str, blocks: int, threads: int, iters: int, device=None,
                     stream=None) -> torch.Tensor:
    """Launch the issue-rate probe for one instruction kind; returns the int64
    [blocks, 3] device tensor of (SM id, start clock, end clock) per CTA (valid
    once the stream has synchronised).  Every thread issues 32 * iters
    instructions."""
    dev = torch.device("cuda") if device is None else device
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    rec = torch.zeros((blocks, 3), dtype=torch.int64, device=dev)
    _check(lib().trit_issue_probe(PROBE_KINDS[kind], blocks, threads, iters,
                                  ctypes.c_void_p(sink.data_ptr()), ctypes.c_void_p(rec.data_ptr()),
                                  _stream(stream)), "trit_issue_probe")
    rec._probe_sink = sink   # keep the sink alive with the record
    return rec


def trit_check_div127() -> int:
    """Number of float32 bit patterns where the library's division by 127 (used
    by every fp32 dequantisation) differs from the IEEE divide; 0 = identical."""
    n = ctypes.c_uint64(0)
    _check(lib().trit_check_div127(ctypes.byref(n)), "trit_check_div127")
    return int(n.value)


def trit_gemv(planes: torch.Tensor, w_scale: float, x_i8: torch.Tensor, x_scale: float,
              K: int, y_i32=None, y_f32=None, err_flag=None, stream=None):
    """One activation row, its scale a host float (the C signature's by-value
    x_scale).  Returns (y_i32 [N], y_f32 [N], err_flag)."""
    if isinstance(x_scale, torch.Tensor):
        raise TypeError("trit_gemv takes x_scale as a float; use trit_gemm for a device scale")
    N = planes.shape[0]
    if y_i32 is None:
        y_i32 = torch.empty(N, dtype=torch.int32, device=planes.device)
    if y_f32 is None:
        y_f32 = torch.empty(N, dtype=torch.float32, device=planes.device)
    err_flag = _err(err_flag, planes.device)
    _check(lib().trit_gemv(_dev(planes, torch.uint8, "planes"), float(w_scale),
                           _dev(x_i8, torch.int8, "x_i8"), float(x_scale),
                           N, K, _dev(y_i32, torch.int32, "y_i32", True),
                           _dev(y_f32, torch.float32, "y_f32", True),
                           _dev(err_flag, torch.int32, "err_flag"), _stream(stream)), "trit_gemv")
    return y_i32, y_f32, err_flag


# trit_proj / trit_qproj flags: the planes were complete before the kernel
# preceding the call on its stream was launched (packed, then synchronised)
PLANES_READY = 1


class ProjList:
    """A prepared host array of trit_proj entries (tensors are kept alive).

    entries: iterables of (planes, w_scale, x_i8, x_scale, K, y_i32, y_f32);
    M is x_i8's row count, N the planes' row count.  planes_ready sets
    PLANES_READY on every entry.
    """

    def __init__(self, entries, planes_ready: bool = False):
        flags = PLANES_READY if planes_ready else 0
        self._keep = []
        items = []
        for planes, w_scale, x_i8, x_scale, K, y_i32, y_f32 in entries:
            M = x_i8.shape[0] if x_i8.dim() == 2 else 1
            items.append(TritProj(
                _dev(planes, torch.uint8, "planes"), _dev(x_i8, torch.int8, "x_i8"),
                _dev(x_scale, torch.float32, "x_scale"),
                _dev(y_i32, torch.int32, "y_i32", True), _dev(y_f32, torch.float32, "y_f32", True),
                M, planes.shape[0], K, float(w_scale), flags))
            self._keep.append((planes, x_i8, x_scale, y_i32, y_f32))
        self.count = len(items)
        self.array = (TritProj * self.count)(*items)


class QProjList:
    """A prepared host array of trit_qproj entries (fused quantise-and-multiply,
    M = 1): (planes, w_scale, x fp32 [K] or [1, K], x_i8 out or None,
    x_scale out or None, y_i32, y_f32).  planes_ready sets PLANES_READY on
    every entry."""

    def __init__(self, entries, planes_ready: bool = False):
        flags = PLANES_READY if planes_ready else 0
        self._keep = []
        items = []
        for planes, w_scale, x, x_i8, x_scale, y_i32, y_f32 in entries:
            K = x.shape[-1]
            items.append(TritQProj(
                _dev(planes, torch.uint8, "planes"), _dev(x, torch.float32, "x"),
                _dev(x_i8, torch.int8, "x_i8", True), _dev(x_scale, torch.float32, "x_scale", True),
                _dev(y_i32, torch.int32, "y_i32", True), _dev(y_f32, torch.float32, "y_f32", True),
                planes.shape[0], K, float(w_scale), flags))
            self._keep.append((planes, x, x_i8, x_scale, y_i32, y_f32))
        self.count = len(items)
        self.array = (TritQProj * self.count)(*items)


class MlpProjList:
    """A prepared host array of trit_mlpproj entries (IntMlp down projections,
    M = 1): (planes, w_scale, a_gate int32 [K], a_up int32 [K], x_scale [1],
    w_gate, w_up, h_i8 out or None, h_scale out or None, y_i32, y_f32)."""

    def __init__(self, entries):
        self._keep = []
        items = []
        for planes, w_scale, a_gate, a_up, x_scale, w_gate, w_up, h_i8, h_scale, y_i32, y_f32 in entries:
            K = a_gate.shape[-1]
            items.append(TritMlpProj(
                _dev(planes, torch.uint8, "planes"), _dev(a_gate, torch.int32, "a_gate"),
                _dev(a_up, torch.int32, "a_up"), _dev(x_scale, torch.float32, "x_scale"),
                float(w_gate), float(w_up), _dev(h_i8, torch.int8, "h_i8", True),
                _dev(h_scale, torch.float32, "h_scale", True),
                _dev(y_i32, torch.int32, "y_i32", True), _dev(y_f32, torch.float32, "y_f32", True),
                planes.shape[0], K, float(w_scale), 0))
            self._keep.append((planes, a_gate, a_up, x_scale, h_i8, h_scale, y_i32, y_f32))
        self.count = len(items)
        self.array = (TritMlpProj * self.count)(*items)


class ActList:
    """A prepared host array of trit_act entries: (x fp32 [M, K], x_i8, x_scale)."""

    def __init__(self, entries):
        self._keep = []
        items = []
        for x, x_i8, x_scale in entries:
            M, K = x.shape
            items.append(TritAct(_dev(x, torch.float32, "x"), _dev(x_i8, torch.int8, "x_i8"),
                                 _dev(x_scale, torch.float32, "x_scale"), M, K))
            self._keep.append((x, x_i8, x_scale))
        self.count = len(items)
        self.array = (TritAct * self.count)(*items)


def trit_gemm_many(plist: ProjList, err_flag: torch.Tensor, stream=None):
    _check(lib().trit_gemm_many(ctypes.cast(plist.array, ctypes.c_void_p), plist.count,
                                _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_gemm_many")


def trit_quant_gemv_many(qlist: QProjList, err_flag: torch.Tensor, stream=None):
    _check(lib().trit_quant_gemv_many(ctypes.cast(qlist.array, ctypes.c_void_p), qlist.count,
                                      _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_quant_gemv_many")


def trit_intmlp_gemv_many(mlist: MlpProjList, err_flag: torch.Tensor, stream=None):
    _check(lib().trit_intmlp_gemv_many(ctypes.cast(mlist.array, ctypes.c_void_p), mlist.count,
                                       _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_intmlp_gemv_many")


def trit_mlp_tmax_bytes(F: int) -> int:
    return int(lib().trit_mlp_tmax_bytes(F))


class MlpBlockList:
    """A prepared host array of trit_mlp_block entries: batch-1 MLP blocks in
    two launches (trit_mlp_gate_up, then trit_mlp_down).  entries: (gate
    planes, up planes, down planes, w_gate, w_up, w_down, x fp32 [K], x_scale
    out [1], a_gate out int32 [F], a_up out int32 [F], tmax workspace (uint8,
    trit_mlp_tmax_bytes(F)), h_i8 out or None, h_scale out or None, y_i32 or
    None, y_f32 or None).  planes_ready sets PLANES_READY on every block."""

    def __init__(self, entries, planes_ready: bool = False):
        flags = PLANES_READY if planes_ready else 0
        self._keep = []
        items = []
        for (gp, upl, dp, w_gate, w_up, w_down, x, x_scale, a_gate, a_up, tmax, h_i8, h_scale,
             y_i32, y_f32) in entries:
            F, Kp = gp.shape[0], gp.shape[1]
            N = dp.shape[0]
            K = x.shape[-1]
            if upl.shape[0] != F or k_pad(K) // 64 != Kp or dp.shape[1] != k_pad(F) // 64:
                raise ValueError("gate, up and down planes do not chain")
            items.append(TritMlpBlock(
                _dev(gp, torch.uint8, "gate_planes"), _dev(upl, torch.uint8, "up_planes"),
                _dev(dp, torch.uint8, "down_planes"), _dev(x, torch.float32, "x"),
                _dev(x_scale, torch.float32, "x_scale"), _dev(a_gate, torch.int32, "a_gate"),
                _dev(a_up, torch.int32, "a_up"), _dev(tmax, torch.uint8, "tmax"),
                _dev(h_i8, torch.int8, "h_i8", True), _dev(h_scale, torch.float32, "h_scale", True),
                _dev(y_i32, torch.int32, "y_i32", True), _dev(y_f32, torch.float32, "y_f32", True),
                K, F, N, float(w_gate), float(w_up), float(w_down), flags))
            self._keep.append((gp, upl, dp, x, x_scale, a_gate, a_up, tmax, h_i8, h_scale,
                               y_i32, y_f32))
        self.count = len(items)
        self.array = (TritMlpBlock * self.count)(*items)


def trit_mlp_gate_up(blist: MlpBlockList, err_flag: torch.Tensor, stream=None):
    _check(lib().trit_mlp_gate_up(ctypes.cast(blist.array, ctypes.c_void_p), blist.count,
                                  _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_mlp_gate_up")


def trit_mlp_down(blist: MlpBlockList, err_flag: torch.Tensor, stream=None):
    _check(lib().trit_mlp_down(ctypes.cast(blist.array, ctypes.c_void_p), blist.count,
                               _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_mlp_down")


def trit_quant_act_many(alist: ActList, err_flag: torch.Tensor, stream=None):
    _check(lib().trit_quant_act_many(ctypes.cast(alist.array, ctypes.c_void_p), alist.count,
                                     _dev(err_flag, torch.int32, "err_flag"), _stream(stream)),
           "trit_quant_act_many")


# ---- BITCOS weights (presence bitmap + compacted signs) ---------------------

def trit_bitcos_pack(w):
    """HOST packer: ternary int8 W [N, K] (numpy array or CPU tensor) -> host
    numpy arrays (bitmap uint64 [N, ceil(K/64)], sign_off uint32 [N+1], signs
    uint32 [sign_off[N] + 2])."""
    import numpy as np
    w = np.ascontiguousarray(w.numpy() if isinstance(w, torch.Tensor) else w, dtype=np.int8)
    N, K = w.shape
    wp = ctypes.c_void_p(w.ctypes.data)
    words = ctypes.c_int64(0)
    _check(lib().trit_bitcos_pack(wp, N, K, None, None, None, ctypes.byref(words)), "trit_bitcos_pack")
    bitmap = np.empty((N, (K + 63) // 64), dtype=np.uint64)
    sign_off = np.empty(N + 1, dtype=np.uint32)
    signs = np.empty(words.value, dtype=np.uint32)
    _check(lib().trit_bitcos_pack(wp, N, K, ctypes.c_void_p(bitmap.ctypes.data),
                                  ctypes.c_void_p(sign_off.ctypes.data),
                                  ctypes.c_void_p(signs.ctypes.data), ctypes.byref(words)),
           "trit_bitcos_pack")
    return bitmap, sign_off, signs


class BitcosWeights:
    """A BITCOS matrix uploaded to the device (the three arrays of trit_bitcos_pack)."""

    def __init__(self, bitmap, sign_off, signs, K: int, device=None):
        dev = torch.device("cuda") if device is None else device
        self.bitmap = torch.from_numpy(bitmap.view("int64")).to(dev)
        self.sign_off = torch.from_numpy(sign_off.view("int32")).to(dev)
        self.signs = torch.from_numpy(signs.view("int32")).to(dev)
        self.N = bitmap.shape[0]
        self.K = int(K)

    @property
    def nbytes(self) -> int:
        return (self.bitmap.numel() * 8 + self.sign_off.numel() * 4 + self.signs.numel() * 4)


class BitcosList:
    """Host array of trit_bitcos_proj entries: (weights, w_scale, x_i8 [K_pad],
    x_scale [1], y_i32 [N] or None, y_f32 [N] or None)."""

    def __init__(self, entries):
        self._keep = []
        items = []
        for W, w_scale, x_i8, x_scale, y_i32, y_f32 in entries:
            items.append(TritBitcosProj(
                _dev(W.bitmap, torch.int64, "bitmap"), _dev(W.sign_off, torch.int32, "sign_off"),
                _dev(W.signs, torch.int32, "signs"), _dev(x_i8, torch.int8, "x_i8"),
                _dev(x_scale, torch.float32, "x_scale"),
                _dev(y_i32, torch.int32, "y_i32", True), _dev(y_f32, torch.float32, "y_f32", True),
                W.N, W.K, W.signs.numel(), float(w_scale), 0))
            self._keep.append((W, x_i8, x_scale, y_i32, y_f32))
        self.count = len(items)
        self.array = (TritBitcosProj * self.count)(*items)


def trit_bitcos_gemv_many(blist: BitcosList, stream=None):
    _check(lib().trit_bitcos_gemv_many(ctypes.cast(blist.array, ctypes.c_void_p), blist.count,
                                       _stream(stream)), "trit_bitcos_gemv_many")


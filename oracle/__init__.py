"""CPU oracle for the ternary bit-plane select-accumulate path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by the CPU-baseline leg of ``bench.py``.  The product package never imports
it, and it shares no code with the CUDA library.

The arithmetic lives in ``trit_oracle.c`` (plain C, single-threaded, bit-by-bit
decode, int64 accumulation); this module compiles it with gcc and wraps it with
numpy arrays.  Every function cites the passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "trit_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

# Row / call error bits returned by the C code.
P1 = 1
P2 = 2
NOT_TERNARY = 4
NONFINITE = 8
OVERFLOW = 32


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (no fast-math,
    no floating-point contraction) and return its path."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        tmp = _OUT + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
             "-fno-fast-math", "-o", tmp, _SRC, "-lm"],
            check=True)
        os.replace(tmp, _OUT)
    return _OUT


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p = ctypes.c_int64, ctypes.c_void_p
            lib.oracle_beats_per_row.restype = i64
            lib.oracle_beats_per_row.argtypes = [i64]
            lib.oracle_payload_bytes.restype = i64
            lib.oracle_payload_bytes.argtypes = [i64, i64]
            lib.oracle_pack.argtypes = [p, i64, i64, p, p]
            lib.oracle_verify.argtypes = [p, i64, i64, p]
            lib.oracle_unpack.argtypes = [p, i64, i64, p, p]
            lib.oracle_quant.argtypes = [p, i64, i64, i64, p, p, p]
            lib.oracle_gemm.argtypes = [p, ctypes.c_float, p, i64, p, i64, i64, i64, p, i64,
                                        p, p, p, p]
            lib.oracle_gemm_popcount.argtypes = [p, p, i64, i64, i64, i64, p]
            lib.oracle_quant_folded.argtypes = [p, p, i64, i64, ctypes.c_double, i64, p, p, p, p]
            lib.oracle_intmlp_quant.argtypes = [p, p, i64, i64, i64, ctypes.c_float,
                                                ctypes.c_float, p, i64, p, p]
            lib.oracle_bitcos_pack_flat.argtypes = [p, i64, p, p, p]
            lib.oracle_bitcos_unpack_flat.argtypes = [p, p, i64, p]
            lib.oracle_bitcos_blocked_words.restype = i64
            lib.oracle_bitcos_blocked_words.argtypes = [p, i64, i64]
            lib.oracle_bitcos_pack_blocked.argtypes = [p, i64, i64, p, p, p]
            lib.oracle_bitcos_gemv.argtypes = [p, p, p, i64, i64, ctypes.c_float, p,
                                               ctypes.c_float, p, i64, p, p]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def beats_per_row(cols: int) -> int:
    return int(_load().oracle_beats_per_row(cols))


def payload_bytes(rows: int, cols: int) -> int:
    return int(_load().oracle_payload_bytes(rows, cols))


class OracleReject(ValueError):
    """The oracle rejected its input; ``code`` is the error bit mask and
    ``where`` the offending index (or None)."""

    def __init__(self, code: int, where=None):
        super().__init__(f"oracle rejected input: code={code} where={where}")
        self.code = code
        self.where = where


def pack(w: np.ndarray) -> np.ndarray:
    """int8 ternary (rows x cols) -> payload uint8 [rows, beats_per_row, 16]."""
    w = np.ascontiguousarray(w, dtype=np.int8)
    rows, cols = w.shape
    out = np.empty((rows, beats_per_row(cols), 16), dtype=np.uint8)
    bad = np.full(1, -1, dtype=np.int64)
    rc = _load().oracle_pack(_ptr(w), rows, cols, _ptr(out), _ptr(bad))
    if rc:
        raise OracleReject(rc, int(bad[0]))
    return out


def unpack(payload: np.ndarray, cols: int) -> np.ndarray:
    payload = np.ascontiguousarray(payload, dtype=np.uint8)
    rows = payload.shape[0]
    w = np.zeros((rows, cols), dtype=np.int8)
    bad = np.full(1, -1, dtype=np.int64)
    rc = _load().oracle_unpack(_ptr(payload), rows, cols, _ptr(w), _ptr(bad))
    if rc:
        raise OracleReject(rc, int(bad[0]))
    return w


def verify(payload: np.ndarray, cols: int):
    """Return (kinds, first): kinds is the OR of P1/P2 found (0 = clean) and
    first the smallest offending bit position (row*B + beat)*64 + k, or -1."""
    payload = np.ascontiguousarray(payload, dtype=np.uint8)
    first = np.full(1, -1, dtype=np.int64)
    kinds = _load().oracle_verify(_ptr(payload), payload.shape[0], cols, _ptr(first))
    return int(kinds), int(first[0])


def quant(x: np.ndarray, ldq: int | None = None):
    """fp32 (M x K) -> (q int8 [M, ldq], scale fp32 [M], row_err uint8 [M])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    M, K = x.shape
    if ldq is None:
        ldq = beats_per_row(K) * 64
    q = np.empty((M, ldq), dtype=np.int8)
    s = np.empty(M, dtype=np.float32)
    e = np.empty(M, dtype=np.uint8)
    _load().oracle_quant(_ptr(x), M, K, ldq, _ptr(q), _ptr(s), _ptr(e))
    return q, s, e


def gemm(payload: np.ndarray, w_scale: float, x_i8: np.ndarray, x_scale: np.ndarray, K: int,
         rows=None):
    """y = W x for the selected rows (all when rows is None).

    x_i8 is [M, ldx] int8 (only columns < K are read), x_scale [M] fp32.
    Returns (y_i32 [M, nsel], y_f32 [M, nsel], row_err [nsel]).
    """
    payload = np.ascontiguousarray(payload, dtype=np.uint8)
    x_i8 = np.ascontiguousarray(x_i8, dtype=np.int8)
    if x_i8.ndim == 1:
        x_i8 = x_i8[None, :]
    x_scale = np.ascontiguousarray(np.atleast_1d(x_scale), dtype=np.float32)
    N = payload.shape[0]
    M, ldx = x_i8.shape
    assert ldx >= K and x_scale.shape[0] == M
    if rows is None:
        sel, nsel, psel = None, N, None
    else:
        sel = np.ascontiguousarray(rows, dtype=np.int64)
        nsel, psel = sel.shape[0], _ptr(sel)
    y = np.empty((M, nsel), dtype=np.int32)
    yf = np.empty((M, nsel), dtype=np.float32)
    err = np.empty(nsel, dtype=np.uint8)
    scratch = np.empty(max(K, 1), dtype=np.int8)
    rc = _load().oracle_gemm(_ptr(payload), ctypes.c_float(w_scale), _ptr(x_i8), ldx,
                             _ptr(x_scale), M, N, K, psel, nsel, _ptr(y), _ptr(yf), _ptr(err),
                             _ptr(scratch))
    if rc & 64:
        raise ValueError("oracle_gemm: bad argument")
    return y, yf, err


def gemm_popcount(payload: np.ndarray, x_i8: np.ndarray, K: int) -> np.ndarray:
    """The bit-serial popcount evaluation of y (int32 [M, N])."""
    payload = np.ascontiguousarray(payload, dtype=np.uint8)
    x_i8 = np.ascontiguousarray(x_i8, dtype=np.int8)
    if x_i8.ndim == 1:
        x_i8 = x_i8[None, :]
    M, ldx = x_i8.shape
    N = payload.shape[0]
    y = np.empty((M, N), dtype=np.int32)
    rc = _load().oracle_gemm_popcount(_ptr(payload), _ptr(x_i8), ldx, M, N, K, _ptr(y))
    if rc:
        raise OracleReject(rc)
    return y


def quant_folded(x: np.ndarray, g: np.ndarray, eps: float, ldq: int | None = None):
    """Folded normalisation + quantisation: codes of x (.) g, scale absmax/rms.
    Returns (q int8 [M, ldq], scale fp32 [M], row_err uint8 [M])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    g = np.ascontiguousarray(g, dtype=np.float32)
    M, K = x.shape
    assert g.shape == (K,)
    if ldq is None:
        ldq = beats_per_row(K) * 64
    q = np.empty((M, ldq), dtype=np.int8)
    s = np.empty(M, dtype=np.float32)
    e = np.empty(M, dtype=np.uint8)
    u = np.empty(K, dtype=np.float32)
    _load().oracle_quant_folded(_ptr(x), _ptr(g), M, K, float(eps), ldq, _ptr(q), _ptr(s),
                                _ptr(e), _ptr(u))
    return q, s, e


def intmlp_quant(a_g: np.ndarray, a_u: np.ndarray, w_g: float, w_u: float, x_scale,
                 ldq: int | None = None):
    """IntMlp + absmax quantisation of the next projection's input.
    a_g, a_u int32 [M, N]; returns (q int8 [M, ldq], h_scale fp32 [M])."""
    a_g = np.ascontiguousarray(a_g, dtype=np.int32)
    a_u = np.ascontiguousarray(a_u, dtype=np.int32)
    if a_g.ndim == 1:
        a_g, a_u = a_g[None, :], a_u[None, :]
    M, N = a_g.shape
    assert a_u.shape == (M, N)
    xs = np.ascontiguousarray(np.atleast_1d(x_scale), dtype=np.float32)
    if ldq is None:
        ldq = beats_per_row(N) * 64
    q = np.empty((M, ldq), dtype=np.int8)
    h = np.empty(M, dtype=np.float32)
    _load().oracle_intmlp_quant(_ptr(a_g), _ptr(a_u), M, N, N, ctypes.c_float(w_g),
                                ctypes.c_float(w_u), _ptr(xs), ldq, _ptr(q), _ptr(h))
    return q, h


# ---- BITCOS ("BITCOS: Intel's Ternary LLM Weight Format Goes Below 1.58 Bits"
# ---- -- A bitmap and a sign) ------------------------------------------------

def bitcos_pack_flat(q: np.ndarray):
    """Flat presence bitmap and sign vector of the ternary codes q (any shape,
    taken in C order).  Returns (bitmap uint8 [ceil(n/8)], signs uint8
    [ceil(nnz/8)])."""
    q = np.ascontiguousarray(q, dtype=np.int8).reshape(-1)
    n = q.shape[0]
    bitmap = np.empty((n + 7) // 8, dtype=np.uint8)
    signs = np.empty(max((n + 7) // 8, 1), dtype=np.uint8)
    nnz = np.zeros(1, dtype=np.int64)
    rc = _load().oracle_bitcos_pack_flat(_ptr(q), n, _ptr(bitmap), _ptr(signs), _ptr(nnz))
    if rc:
        raise OracleReject(rc)
    return bitmap, signs[:(int(nnz[0]) + 7) // 8].copy()


def bitcos_unpack_flat(bitmap: np.ndarray, signs: np.ndarray, n: int) -> np.ndarray:
    bitmap = np.ascontiguousarray(bitmap, dtype=np.uint8)
    signs = np.ascontiguousarray(signs, dtype=np.uint8)
    if signs.size == 0:
        signs = np.zeros(1, dtype=np.uint8)
    q = np.empty(n, dtype=np.int8)
    _load().oracle_bitcos_unpack_flat(_ptr(bitmap), _ptr(signs), n, _ptr(q))
    return q


def bitcos_pack_blocked(w: np.ndarray):
    """Blocked BITCOS form of a [rows, cols] ternary matrix: (bitmap uint64
    [rows, ceil(cols/64)], sign_off uint32 [rows+1], signs uint32
    [sign_off[-1] + 2])."""
    w = np.ascontiguousarray(w, dtype=np.int8)
    rows, cols = w.shape
    lib = _load()
    words = int(lib.oracle_bitcos_blocked_words(_ptr(w), rows, cols))
    bitmap = np.empty((rows, (cols + 63) // 64), dtype=np.uint64)
    sign_off = np.empty(rows + 1, dtype=np.uint32)
    signs = np.empty(words + 2, dtype=np.uint32)
    rc = lib.oracle_bitcos_pack_blocked(_ptr(w), rows, cols, _ptr(bitmap), _ptr(sign_off),
                                        _ptr(signs))
    if rc:
        raise OracleReject(rc)
    return bitmap, sign_off, signs


def bitcos_gemv(bitmap: np.ndarray, sign_off: np.ndarray, signs: np.ndarray, cols: int,
                w_scale: float, x_i8: np.ndarray, x_scale: float, rows=None):
    """y = W x (one activation row) from the blocked form; returns (y_i32, y_f32)
    for the selected rows (all when rows is None)."""
    bitmap = np.ascontiguousarray(bitmap, dtype=np.uint64)
    sign_off = np.ascontiguousarray(sign_off, dtype=np.uint32)
    signs = np.ascontiguousarray(signs, dtype=np.uint32)
    x_i8 = np.ascontiguousarray(x_i8, dtype=np.int8).reshape(-1)
    assert x_i8.shape[0] >= cols
    nrows = bitmap.shape[0]
    if rows is None:
        sel, nsel, psel = None, nrows, None
    else:
        sel = np.ascontiguousarray(rows, dtype=np.int64)
        nsel, psel = sel.shape[0], _ptr(sel)
    y = np.empty(nsel, dtype=np.int32)
    yf = np.empty(nsel, dtype=np.float32)
    rc = _load().oracle_bitcos_gemv(_ptr(bitmap), _ptr(sign_off), _ptr(signs), nrows, cols,
                                    ctypes.c_float(w_scale), _ptr(x_i8), ctypes.c_float(x_scale),
                                    psel, nsel, _ptr(y), _ptr(yf))
    if rc & 64:
        raise ValueError("oracle_bitcos_gemv: bad argument")
    return y, yf


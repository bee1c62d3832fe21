"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every entry point include/trit.h declares; the ctypes structs match
the header's layout; argument errors are rejected before anything touches a
device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def trit():
    from bit_plane_select_gb300 import build
    build.build()
    import bit_plane_select_gb300 as t
    return t


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"TRIT_API\s+[\w\s\*]+?\b(trit_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("trit_pack", "trit_unpack", "trit_verify", "trit_quant_act", "trit_gemv",
                     "trit_gemm", "trit_gemm_many", "trit_quant_act_many",
                     "trit_quant_gemv_many", "trit_gemm_noalloc", "trit_file_open",
                     "trit_file_open_memory", "trit_file_verify", "trit_file_upload",
                     "trit_fnv1a64", "trit_bitcos_pack", "trit_bitcos_gemv_many"):
        assert required in names


def test_library_exports_every_declared_symbol(trit):
    lib = ctypes.CDLL(trit.library_path())
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert trit.lib().trit_abi_version() == 4


def test_struct_layouts(trit):
    assert ctypes.sizeof(trit.TritProj) == 72
    assert trit.TritProj.w_scale.offset == 64
    assert ctypes.sizeof(trit.TritAct) == 40
    assert ctypes.sizeof(trit.TritQProj) == 72 and trit.TritQProj.w_scale.offset == 64
    assert ctypes.sizeof(trit.TritMlpProj) == 96
    assert ctypes.sizeof(trit.TritBitcosProj) == 88
    assert ctypes.sizeof(trit.TritMlpBlock) == 136


def test_struct_layouts_match_the_c_compiler(trit, tmp_path):
    """Every field offset of the ctypes mirrors equals what the C compiler lays
    out from include/trit.h."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"trit_proj": trit.TritProj, "trit_qproj": trit.TritQProj,
               "trit_act": trit.TritAct, "trit_mlpproj": trit.TritMlpProj,
               "trit_bitcos_proj": trit.TritBitcosProj, "trit_mlp_block": trit.TritMlpBlock}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "trit.h"', "int main(void) {"]
    for cname, cls in structs.items():
        lines.append(f'printf("{cname} size %zu\\n", sizeof({cname}));')
        for fname, _ in cls._fields_:
            lines.append(f'printf("{cname} {fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    got = {}
    for line in out:
        if line:
            c, f, v = line.split()
            got[(c, f)] = int(v)
    for cname, cls in structs.items():
        assert got[(cname, "size")] == ctypes.sizeof(cls), cname
        for fname, _ in cls._fields_:
            assert got[(cname, fname)] == getattr(cls, fname).offset, (cname, fname)


def test_mlp_block_validation(trit):
    """trit_mlp_gate_up / trit_mlp_down reject bad blocks before touching a
    device; the partials workspace is 144 bytes per 32 gate/up rows."""
    L = trit.lib()
    assert L.trit_mlp_tmax_bytes(6912) == 144 * 216
    assert L.trit_mlp_tmax_bytes(1) == 144 and L.trit_mlp_tmax_bytes(33) == 288
    assert L.trit_mlp_tmax_bytes(0) == 0
    p, null, odd = ctypes.c_void_p(1 << 16), None, ctypes.c_void_p((1 << 16) + 4)
    s = ctypes.c_void_p(None)
    B = trit.TritMlpBlock

    def blk(**kw):
        a = dict(gate_planes=p, up_planes=p, down_planes=p, x=p, x_scale=p, a_gate=p, a_up=p,
                 tmax=p, h_i8=null, h_scale=null, y_i32=p, y_f32=p, K=2560, F=6912, N=2560,
                 w_gate=1.0, w_up=1.0, w_down=1.0, flags=0)
        a.update(kw)
        return B(**a)

    for bad, code in [(blk(tmax=null), 1), (blk(a_gate=odd), 1), (blk(y_i32=null, y_f32=null), 1),
                      (blk(flags=2), 1), (blk(x=null), 1), (blk(F=0), 2), (blk(K=trit.MAX_FUSED_K + 1), 2),
                      (blk(F=trit.MAX_FUSED_K + 1), 2), (blk(N=0), 2), (blk(w_up=0.0), 4),
                      (blk(w_down=float("nan")), 4)]:
        lst = (B * 2)(blk(), bad)
        for fn in (L.trit_mlp_gate_up, L.trit_mlp_down):
            assert fn(ctypes.cast(lst, ctypes.c_void_p), 2, p, s) == code
    lst = (B * 1)(blk())
    assert L.trit_mlp_gate_up(ctypes.cast(lst, ctypes.c_void_p), 0, p, s) == 1
    assert L.trit_mlp_down(ctypes.cast(lst, ctypes.c_void_p), 1, null, s) == 1


def test_payload_bytes(trit):
    assert trit.payload_bytes(2560, 2560) == 1638400
    assert trit.payload_bytes(2, 3) == 32
    assert trit.payload_bytes(0, 3) == -1
    assert trit.payload_bytes(1, 1 << 24) == -1


def test_status_strings(trit):
    L = trit.lib()
    assert L.trit_status_string(0) == b"TRIT_OK"
    assert L.trit_status_string(2).startswith(b"TRIT_E_SHAPE")
    assert L.trit_status_string(9).startswith(b"TRIT_E_VALUE")


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="uses fake pointers; only run where no GPU can be reached")
def test_argument_errors_are_rejected_on_the_host(trit):
    """Every case here is invalid by construction, so the library must return
    before any CUDA call; nothing is enqueued."""
    L = trit.lib()
    p = ctypes.c_void_p(0x10000)       # a 16-byte-aligned fake address, never dereferenced
    odd = ctypes.c_void_p(0x10001)
    null = ctypes.c_void_p(0)
    s = null
    # trit_pack(w, N, K, w_scale, planes, scale_out, err, stream)
    assert L.trit_pack(null, 4, 64, 1.0, p, null, p, s) == 1
    assert L.trit_pack(p, 4, 64, 1.0, odd, null, p, s) == 1
    assert L.trit_pack(p, 0, 64, 1.0, p, null, p, s) == 2
    assert L.trit_pack(p, 4, 1 << 24, 1.0, p, null, p, s) == 2
    assert L.trit_pack(p, 4, 64, float("nan"), p, null, p, s) == 4
    assert L.trit_pack(p, 4, 64, 0.0, p, null, p, s) == 4
    assert L.trit_pack(p, 4, 64, -1.0, p, null, p, s) == 4
    # trit_gemm(planes, w_scale, x, x_scale, M, N, K, y_i32, y_f32, err, stream)
    assert L.trit_gemm(p, 1.0, p, p, 1, 8, 64, null, null, p, s) == 1
    assert L.trit_gemm(p, 1.0, p, p, 0, 8, 64, p, p, p, s) == 2
    assert L.trit_gemm(p, 1.0, p, p, 1, 8, 0, p, p, p, s) == 2
    assert L.trit_gemm(p, float("inf"), p, p, 1, 8, 64, p, p, p, s) == 4
    assert L.trit_gemm(p, 1.0, odd, p, 1, 8, 64, p, p, p, s) == 1
    assert L.trit_gemm(p, 1.0, p, p, 1, 8, 64, p, p, null, s) == 1
    assert L.trit_gemm_many(null, 1, p, s) == 1
    lst = (trit.TritProj * 2)(trit.TritProj(p, p, p, p, p, 1, 8, 64, 1.0, 0),
                              trit.TritProj(p, p, p, p, p, 1, 8, 64, 1.0, 7))
    assert L.trit_gemm_many(ctypes.cast(lst, ctypes.c_void_p), 2, p, s) == 1   # unknown flag bits
    assert L.trit_gemm_many(ctypes.cast(lst, ctypes.c_void_p), 0, p, s) == 1
    # trit_quant_act(x, M, K, x_i8, x_scale, err, stream)
    assert L.trit_quant_act(p, 2, 0, p, p, p, s) == 2
    assert L.trit_quant_act(p, 2, 10, odd, p, p, s) == 1
    # trit_verify(planes, N, K, err, first_bad, stream)
    assert L.trit_verify(p, 2, 10, null, null, s) == 1
    assert L.trit_verify(p, 2, 10, p, ctypes.c_void_p(0x10004), s) == 1
    # trit_bitcos_gemv_many(list, count, stream)
    B = trit.TritBitcosProj
    assert L.trit_bitcos_gemv_many(null, 1, s) == 1
    ok = B(p, p, p, p, p, p, p, 8, 64, 10, 1.0, 0)
    cases = [(B(p, p, p, p, p, p, p, 8, 64, 10, 1.0, 3), 1),              # reserved
             (B(ctypes.c_void_p(0x10008), p, p, p, p, p, p, 8, 64, 10, 1.0, 0), 1),   # bitmap align
             (B(p, p, p, p, p, null, null, 8, 64, 10, 1.0, 0), 1),        # no output
             (B(p, p, p, p, p, p, p, 8, trit.BITCOS_MAX_K + 1, 10, 1.0, 0), 2),
             (B(p, p, p, p, p, p, p, 0, 64, 10, 1.0, 0), 2),
             (B(p, p, p, p, p, p, p, 8, 64, 1, 1.0, 0), 2),                # sign_words < 2
             (B(p, p, p, p, p, p, p, 8, 64, 10, float("nan"), 0), 4)]
    for bad, code in cases:
        lst = (B * 2)(ok, bad)
        assert L.trit_bitcos_gemv_many(ctypes.cast(lst, ctypes.c_void_p), 2, s) == code
    lst = (B * 1)(ok)
    assert L.trit_bitcos_gemv_many(ctypes.cast(lst, ctypes.c_void_p), 0, s) == 1


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="uses fake pointers; only run where no GPU can be reached")
def test_argument_errors_of_the_other_entry_points(trit):
    """The entry points the test above leaves out: each case is invalid by
    construction and must be refused on the host before any CUDA call."""
    L = trit.lib()
    p = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10001)
    null = ctypes.c_void_p(0)
    s = null
    nan = float("nan")
    # trit_unpack(planes, N, K, w, err, stream)
    assert L.trit_unpack(p, 4, 64, null, p, s) == 1
    assert L.trit_unpack(odd, 4, 64, p, p, s) == 1
    assert L.trit_unpack(p, 0, 64, p, p, s) == 2
    # trit_gemv(planes, w_scale, x, x_scale BY VALUE, N, K, y_i32, y_f32, err, stream)
    inf = float("inf")
    assert L.trit_gemv(p, 1.0, p, 1.0, 8, 64, null, null, p, s) == 1
    assert L.trit_gemv(p, 1.0, odd, 1.0, 8, 64, p, p, p, s) == 1
    assert L.trit_gemv(p, 1.0, p, 1.0, 8, 64, p, p, null, s) == 1
    assert L.trit_gemv(p, 1.0, p, 1.0, 8, 0, p, p, p, s) == 2
    assert L.trit_gemv(p, 1.0, p, 1.0, 0, 64, p, p, p, s) == 2
    assert L.trit_gemv(p, nan, p, 1.0, 8, 64, p, p, p, s) == 4
    for bad_xs in (nan, inf, -1.0):
        assert L.trit_gemv(p, 1.0, p, bad_xs, 8, 64, p, p, p, s) == 4
    # valid arguments pass the host checks and stop at the device check
    # (TRIT_E_CUDA or TRIT_E_DEVICE where no sm_103 GPU can be reached)
    for good_xs in (0.0, 1.0, 3e38):
        assert L.trit_gemv(p, 1.0, p, good_xs, 8, 64, p, p, p, s) in (6, 7)
    # trit_quant_act_many(list, count, err, stream)
    A = trit.TritAct
    assert L.trit_quant_act_many(null, 1, p, s) == 1
    acts = (A * 2)(A(p, p, p, 2, 64), A(p, p, p, 2, 0))
    assert L.trit_quant_act_many(ctypes.cast(acts, ctypes.c_void_p), 2, p, s) == 2
    acts = (A * 1)(A(p, odd, p, 2, 64))
    assert L.trit_quant_act_many(ctypes.cast(acts, ctypes.c_void_p), 1, p, s) == 1
    assert L.trit_quant_act_many(ctypes.cast(acts, ctypes.c_void_p), 0, p, s) == 1
    # trit_quant_gemv_many(list, count, err, stream)
    Q = trit.TritQProj
    good_q = Q(p, p, p, p, p, p, 8, 64, 1.0, 0)
    for bad, code in [(Q(p, p, p, p, p, p, 8, 64, 1.0, 2), 1),   # unknown flag bit
                      (Q(p, null, p, p, p, p, 8, 64, 1.0, 0), 1),
                      (Q(p, p, odd, p, p, p, 8, 64, 1.0, 0), 1),
                      (Q(p, p, p, p, p, p, 8, trit.MAX_FUSED_K + 1, 1.0, 0), 2),
                      (Q(p, p, p, p, p, p, 8, 64, 0.0, 0), 4)]:
        lst = (Q * 2)(good_q, bad)
        assert L.trit_quant_gemv_many(ctypes.cast(lst, ctypes.c_void_p), 2, p, s) == code
    # trit_intmlp_gemv_many(list, count, err, stream)
    Mp = trit.TritMlpProj
    good_m = Mp(p, p, p, p, 1.0, 1.0, p, p, p, p, 8, 64, 1.0, 0)
    for bad, code in [(Mp(p, p, p, p, 1.0, 1.0, p, p, p, p, 8, 64, 1.0, 2), 1),
                      (Mp(p, p, p, p, 1.0, 1.0, odd, p, p, p, 8, 64, 1.0, 0), 1),
                      (Mp(p, p, p, p, 1.0, 1.0, p, p, null, null, 8, 64, 1.0, 0), 1),
                      (Mp(p, p, p, p, 1.0, 1.0, p, p, p, p, 8, trit.MAX_FUSED_K + 1, 1.0, 0), 2),
                      (Mp(p, p, p, p, nan, 1.0, p, p, p, p, 8, 64, 1.0, 0), 4),
                      (Mp(p, p, p, p, 1.0, -1.0, p, p, p, p, 8, 64, 1.0, 0), 4)]:
        lst = (Mp * 2)(good_m, bad)
        assert L.trit_intmlp_gemv_many(ctypes.cast(lst, ctypes.c_void_p), 2, p, s) == code
    # trit_quant_act_folded(x, gain, M, K, eps, x_i8, x_scale, err, stream)
    assert L.trit_quant_act_folded(p, null, 2, 64, 1e-6, p, p, p, s) == 1
    assert L.trit_quant_act_folded(p, p, 2, 0, 1e-6, p, p, p, s) == 2
    assert L.trit_quant_act_folded(p, p, 2, 64, -1.0, p, p, p, s) == 4
    # trit_intmlp_quant(a_gate, a_up, M, N, w_gate, w_up, x_scale, h_i8, h_scale, stream)
    assert L.trit_intmlp_quant(p, p, 1, 64, 1.0, 1.0, p, odd, p, s) == 1
    assert L.trit_intmlp_quant(p, p, 1, 0, 1.0, 1.0, p, p, p, s) == 2
    assert L.trit_intmlp_quant(p, p, 1, 64, 1.0, 0.0, p, p, p, s) == 4
    # trit_gemm_noalloc(planes, w_scale, x, x_scale, M, N, K, y_i32, y_f32, err, stream)
    assert L.trit_gemm_noalloc(p, 1.0, p, p, 1, 8, 64, p, p, null, s) == 1
    assert L.trit_gemm_noalloc(p, 1.0, p, p, 1, 8, 0, p, p, p, s) == 2
    assert L.trit_gemm_noalloc(p, 0.0, p, p, 1, 8, 64, p, p, p, s) == 4
    # trit_read_probe(buf, bytes, sink, stream), trit_check_div127(mismatches)
    assert L.trit_read_probe(p, 8, p, s) == 1
    assert L.trit_read_probe(p, 17, p, s) == 1
    assert L.trit_read_probe(p, 64, null, s) == 1
    assert L.trit_check_div127(None) == 1


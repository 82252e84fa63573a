"""The C-ABI library (liblq.so) loads on the host, exports every entry point
that include/lq.h declares, and validates arguments before touching the GPU
(these calls return before any CUDA call, so they run without a GPU)."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "lq.h")


@pytest.fixture(scope="module")
def lq():
    import block_quantized_weight_super_gb300 as pkg
    from block_quantized_weight_super_gb300 import build
    build.build()
    pkg.lib()
    return pkg


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lq_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_api():
    names = declared_functions()
    for n in ["lq_dequant", "lq_matvec", "lq_qkv_mixed", "lq_pack_gate_up", "lq_ffn_gate_up_act",
              "lq_moe_workspace_bytes", "lq_moe_ffn"]:
        assert n in names


def test_library_exports_every_declared_symbol(lq):
    L = C.CDLL(lq.LIB_PATH)
    for n in declared_functions():
        assert hasattr(L, n), n
    assert sorted(lq.EXPORTS) == declared_functions()


def _declared_params():
    """(name, [C parameter types]) of every function lq.h declares."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, args in re.findall(r"\b(lq_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", src):
        args = args.strip()
        out[name] = [] if args in ("", "void") else [a.strip() for a in args.split(",")]
    return out


def _ctype_class(c_param):
    """the ctypes type a C parameter must be passed as"""
    t = re.sub(r"\b[A-Za-z_0-9]+$", "", c_param).strip()   # drop the parameter name
    if "*" in t or t == "lq_stream_t":
        return "pointer"
    return {"int": C.c_int, "int64_t": C.c_int64, "uint64_t": C.c_uint64, "size_t": C.c_size_t,
            "float": C.c_float}[t.replace("const ", "")]


def test_binding_signatures_match_header(lq):
    """every ctypes signature of the binding passes each argument as the type
    lq.h declares (a count or width mismatch would pass garbage silently)"""
    L = lq.lib()
    decl = _declared_params()
    assert sorted(decl) == declared_functions()
    for name, params in decl.items():
        argtypes = getattr(L, name).argtypes or []
        assert len(argtypes) == len(params), (name, len(argtypes), len(params))
        for i, (c_param, ct) in enumerate(zip(params, argtypes)):
            want = _ctype_class(c_param)
            if want == "pointer":
                assert ct is C.c_void_p or ct is C.c_char_p or hasattr(ct, "contents") or \
                    getattr(ct, "_type_", None) is not None and issubclass(ct, C._Pointer), (name, i, c_param, ct)
            else:
                assert ct is want, (name, i, c_param, ct)


def test_format_facts(lq):
    assert lq.lq_block_bytes(1) == 144 and lq.lq_block_elems(1) == 256
    assert lq.lq_block_bytes(2) == 210 and lq.lq_block_elems(2) == 256
    assert lq.lq_block_bytes(3) == 34 and lq.lq_block_elems(3) == 32
    assert lq.lq_block_bytes(9) == 0 and lq.lq_block_elems(0) == 0
    assert lq.lq_row_bytes(1, 2560) == 1440
    assert lq.lq_row_bytes(2, 2560) == 2100
    assert lq.lq_row_bytes(3, 96) == 102
    assert lq.lq_row_bytes(3, 100) == 0


def test_status_strings(lq):
    for s in range(8):
        assert lq.lq_status_str(s).startswith("LQ_")


# Arguments rejected on the host: no CUDA call is made on these paths.
FAKE = 0x10000      # a 16-byte aligned non-null address never dereferenced here


def _rc(f, *a):
    return getattr(C.CDLL(__import__("block_quantized_weight_super_gb300").LIB_PATH), f)(*a)


def test_matvec_validation(lq):
    L = lq.lib()
    i64 = C.c_int64
    assert L.lq_matvec(1, None, 4, 256, FAKE, FAKE, 1, None) == lq.LQ_EINVAL
    assert L.lq_matvec(1, FAKE, 4, 250, FAKE, FAKE, 1, None) == lq.LQ_ESHAPE
    assert L.lq_matvec(3, FAKE, 4, 48, FAKE, FAKE, 1, None) == lq.LQ_ESHAPE
    assert L.lq_matvec(1, FAKE, 4, 256, FAKE, FAKE, 0, None) == lq.LQ_EINVAL
    assert L.lq_matvec(7, FAKE, 4, 256, FAKE, FAKE, 1, None) == lq.LQ_EINVAL
    assert L.lq_matvec(1, FAKE + 1, 4, 256, FAKE, FAKE, 1, None) == lq.LQ_EALIGN
    assert L.lq_matvec(1, FAKE, 4, 256, FAKE + 2, FAKE, 1, None) == lq.LQ_EALIGN
    assert L.lq_matvec(1, FAKE, 4, 256, FAKE, FAKE + 1, 1, None) == lq.LQ_EALIGN
    assert L.lq_matvec(1, FAKE, 4, 256, None, FAKE, 1, None) == lq.LQ_EINVAL
    assert L.lq_matvec(1, FAKE, -1, 256, FAKE, FAKE, 1, None) == lq.LQ_ESHAPE
    # rows == 0: nothing to do, no launch
    assert L.lq_matvec(1, FAKE, 0, 256, FAKE, FAKE, 1, None) == lq.LQ_OK
    assert "batch" in lq.lq_last_error() or lq.lq_last_error() == ""


def test_softcap_validation(lq):
    L = lq.lib()
    f = lambda cap, x=FAKE: L.lq_matvec_softcap(1, FAKE, 4, 256, x, FAKE, 1, C.c_float(cap), None)
    assert f(0.0) == lq.LQ_EINVAL
    assert f(-30.0) == lq.LQ_EINVAL
    assert f(float("nan")) == lq.LQ_EINVAL
    assert f(float("inf")) == lq.LQ_EINVAL
    assert f(30.0, x=None) == lq.LQ_EINVAL
    assert L.lq_matvec_softcap(1, FAKE, 0, 256, FAKE, FAKE, 1, C.c_float(30.0), None) == lq.LQ_OK   # no rows


def test_other_entry_validation(lq):
    L = lq.lib()
    assert L.lq_dequant(2, FAKE, 3, 100, FAKE, None) == lq.LQ_ESHAPE
    assert L.lq_dequant(2, FAKE, 0, 256, FAKE, None) == lq.LQ_OK
    assert L.lq_ffn_gate_up_act(1, FAKE, 4, 256, FAKE, FAKE, 1, 3, None) == lq.LQ_EINVAL
    assert L.lq_ffn_gate_up_act(1, FAKE, 0, 256, FAKE, FAKE, 1, 1, None) == lq.LQ_OK
    assert L.lq_pack_gate_up(1, FAKE, FAKE, 4, 256, None, None) == lq.LQ_EINVAL
    assert L.lq_qkv_mixed(1, FAKE, 4, 1, FAKE, 4, 2, FAKE, 4, 300, FAKE, FAKE, FAKE, FAKE, 1,
                          None) == lq.LQ_ESHAPE
    assert L.lq_qkv_mixed(1, FAKE, 0, 1, FAKE, 0, 2, FAKE, 0, 256, FAKE, FAKE, FAKE, FAKE, 1,
                          None) == lq.LQ_OK


def test_ffn_validation(lq):
    L = lq.lib()
    ffn = lambda f0, w, f1, wd, inter, hidden, x, h, y, b, act: L.lq_ffn(
        f0, w, f1, wd, inter, hidden, x, h, y, b, act, None)
    assert ffn(1, None, 2, FAKE, 256, 256, FAKE, FAKE, FAKE, 1, 1) == lq.LQ_EINVAL
    assert ffn(1, FAKE, 2, None, 256, 256, FAKE, FAKE, FAKE, 1, 1) == lq.LQ_EINVAL
    assert ffn(1, FAKE, 2, FAKE, 256, 250, FAKE, FAKE, FAKE, 1, 1) == lq.LQ_ESHAPE   # hidden % 256
    assert ffn(1, FAKE, 2, FAKE, 100, 256, FAKE, FAKE, FAKE, 1, 1) == lq.LQ_ESHAPE   # inter % 256 (down cols)
    assert ffn(1, FAKE, 2, FAKE, 0, 256, FAKE, FAKE, FAKE, 1, 1) == lq.LQ_ESHAPE
    assert ffn(1, FAKE, 2, FAKE, 256, 256, FAKE, FAKE, FAKE, 0, 1) == lq.LQ_EINVAL
    assert ffn(1, FAKE, 2, FAKE, 256, 256, FAKE, FAKE, FAKE, 1, 3) == lq.LQ_EINVAL
    assert ffn(1, FAKE, 9, FAKE, 256, 256, FAKE, FAKE, FAKE, 1, 1) == lq.LQ_EINVAL
    assert ffn(1, FAKE, 2, FAKE, 256, 256, FAKE, None, FAKE, 1, 1) == lq.LQ_EINVAL
    assert ffn(1, FAKE, 2, FAKE, 256, 256, FAKE, FAKE + 2, FAKE, 1, 1) == lq.LQ_EALIGN


def test_moe_validation(lq):
    L = lq.lib()
    P = C.c_void_p * 2
    w = P(FAKE, FAKE)
    wp = C.cast(w, C.c_void_p)
    need = lq.lq_moe_workspace_bytes(2, 1, 4, 256, 256)
    assert need > 0
    assert lq.lq_moe_workspace_bytes(0, 1, 4, 256, 256) == 0
    args = lambda E, k, ntok, ws, wsb: L.lq_moe_ffn(FAKE, E, k, 1, wp, wp, wp, 256, 256, FAKE,
                                                   FAKE, ntok, None, None, ws, wsb, None)
    assert args(2, 3, 4, FAKE, need) == lq.LQ_EINVAL        # topk > n_experts
    assert args(2, 0, 4, FAKE, need) == lq.LQ_EINVAL
    assert args(2, 1, 4, FAKE, need - 1) == lq.LQ_EWORKSPACE
    assert args(2, 1, 4, None, need) == lq.LQ_EWORKSPACE
    assert args(2, 1, 4, FAKE + 16, need) == lq.LQ_EALIGN    # workspace 256-aligned
    assert args(2, 1, 0, FAKE, need) == lq.LQ_OK            # no tokens: no launch


def test_moe_ex_validation(lq):
    """The MoE variants' arguments are checked on the host before the
    workspace: shared-expert arrays, their width, the gate without shared
    experts, the weighting flag."""
    L = lq.lib()
    P = C.c_void_p * 2
    w = P(FAKE, FAKE)
    wp = C.cast(w, C.c_void_p)
    need = lq.lq_moe_ffn_ex_workspace_bytes(2, 1, 4, 256, 256, 2, 512)
    assert need > lq.lq_moe_workspace_bytes(2, 1, 4, 256, 256)
    assert lq.lq_moe_ffn_ex_workspace_bytes(2, 1, 4, 256, 256, 0, 0) == lq.lq_moe_workspace_bytes(2, 1, 4, 256, 256)
    assert lq.lq_moe_ffn_ex_workspace_bytes(2, 1, 4, 256, 256, -1, 0) == 0

    def ex(norm=1, ns=2, s1=wp, s3=wp, s2=wp, inter_s=512, gate=FAKE, ws=FAKE, wsb=need, ntok=4):
        return L.lq_moe_ffn_ex(FAKE, 2, 1, norm, 1, wp, wp, wp, 256, 256, ns, s1, s3, s2, inter_s, gate,
                               FAKE, FAKE, ntok, None, None, ws, wsb, None)
    assert ex(norm=2) == lq.LQ_EINVAL
    assert ex(ns=-1) == lq.LQ_EINVAL
    assert ex(ns=lq.LQ_MOE_MAX_SHARED + 1) == lq.LQ_EINVAL
    assert ex(s1=None) == lq.LQ_EINVAL
    assert ex(s2=None) == lq.LQ_EINVAL
    assert ex(inter_s=500) == lq.LQ_ESHAPE              # not a multiple of the Q4_K block
    assert ex(ns=0, gate=FAKE) == lq.LQ_EINVAL          # a gate without shared experts
    assert ex(gate=FAKE + 2) == lq.LQ_EALIGN
    assert ex(wsb=need - 1) == lq.LQ_EWORKSPACE
    assert ex(ws=FAKE + 16) == lq.LQ_EALIGN
    assert ex(ntok=0, ws=None, wsb=0) == lq.LQ_OK        # no tokens: nothing checked past the shapes, no launch


def test_moe_static_validates_before_the_scratch_size(lq):
    """Invalid arguments are reported as such even when the shape would also
    exceed the static scratch (argument errors come first)."""
    L = lq.lib()
    P = C.c_void_p * 2
    w = P(FAKE, FAKE)
    wp = C.cast(w, C.c_void_p)
    st = lambda E, k, fmt, hidden, inter, ntok, x=FAKE: L.lq_moe_ffn_static(
        FAKE, E, k, fmt, wp, wp, wp, hidden, inter, x, FAKE, ntok, None, None, None)
    big = 4096                                          # 2 experts x 4096 tokens: far over 4 MiB
    assert st(2, 3, 1, 4096, 14336, big) == lq.LQ_EINVAL     # topk > n_experts
    assert st(2, 1, 9, 4096, 14336, big) == lq.LQ_EINVAL     # unknown format
    assert st(2, 1, 1, 4096, 14300, big) == lq.LQ_ESHAPE     # inter not a block multiple
    assert st(2, 1, 1, 4096, 14336, 8, x=FAKE + 2) == lq.LQ_EALIGN
    assert st(2, 1, 1, 4096, 14336, 1000) == lq.LQ_EWORKSPACE


def test_fused_norm_and_act_validation(lq):
    """The input-norm and activated-input entry points check epsilon, the
    norm weight, and that the written intermediate does not overlap the
    input, before any launch."""
    L = lq.lib()
    n, cols = 64, 512
    qkv = lambda x=FAKE, w=FAKE, eps=1e-6, xn=FAKE + (1 << 20): L.lq_qkv_mixed_rmsnorm(
        1, FAKE, n, 1, FAKE, n, 2, FAKE, n, cols, x, w, eps, xn, FAKE, FAKE, FAKE, 1, None)
    assert qkv(eps=-1.0) == lq.LQ_EINVAL
    assert qkv(eps=float("nan")) == lq.LQ_EINVAL
    assert qkv(w=None) == lq.LQ_EINVAL
    assert qkv(xn=None) == lq.LQ_EINVAL
    assert qkv(xn=FAKE + 1024) == lq.LQ_EINVAL              # overlaps x (512 floats = 2048 bytes)
    assert qkv(xn=FAKE + 2) == lq.LQ_EALIGN
    gu = lambda eps=1e-6, xn=FAKE + (1 << 20), act=1: L.lq_ffn_gate_up_act_rmsnorm(
        1, FAKE, n, cols, FAKE, FAKE, eps, xn, FAKE, 1, act, None)
    assert gu(eps=float("inf")) == lq.LQ_EINVAL
    assert gu(xn=FAKE) == lq.LQ_EINVAL
    assert gu(act=3) == lq.LQ_EINVAL
    act = lambda h=FAKE + (1 << 20), a=1, gup=FAKE: L.lq_matvec_act(2, FAKE, n, cols, gup, h, FAKE, 1, a, None)
    assert act(a=0) == lq.LQ_EINVAL
    assert act(h=None) == lq.LQ_EINVAL
    assert act(h=FAKE + 4096 - 4) == lq.LQ_EINVAL           # overlaps the 1024-float pair row
    assert act(gup=None) == lq.LQ_EINVAL
    rn = lambda ntok=1, nn=cols, eps=1e-6: L.lq_rmsnorm(FAKE, FAKE, eps, FAKE, ntok, nn, None)
    assert rn(nn=0) == lq.LQ_ESHAPE
    assert rn(ntok=-1) == lq.LQ_ESHAPE
    assert rn(eps=-1e-3) == lq.LQ_EINVAL
    assert rn(ntok=0) == lq.LQ_OK


def test_dense_gemv_validation(lq):
    L = lq.lib()
    f16 = lambda rows=16, cols=64, b=1, W=FAKE, x=FAKE: L.lq_gemv_f16(W, rows, cols, x, FAKE, b, None)
    assert f16(cols=60) == lq.LQ_ESHAPE            # not a multiple of 8 halves
    assert f16(b=0) == lq.LQ_EINVAL
    assert f16(b=9) == lq.LQ_EINVAL
    assert f16(cols=8192, b=8) == lq.LQ_ESHAPE     # x staging over 200 KB
    assert f16(W=None) == lq.LQ_EINVAL
    assert f16(W=FAKE + 8) == lq.LQ_EALIGN
    assert f16(x=FAKE + 4) == lq.LQ_EALIGN
    assert f16(rows=0) == lq.LQ_OK
    assert L.lq_gemv_f32(FAKE, 16, 62, FAKE, FAKE, 1, None) == lq.LQ_ESHAPE


def test_gemm_validation(lq):
    L = lq.lib()
    need = lq.lq_gemm_workspace_bytes(64, 128, 2560)
    assert need >= 64 * 2560 * 4
    # the tcgen05 kernel's x image is padded to whole 128-row tiles, plus s_n and a scale per weight row
    assert lq.lq_gemm_workspace_bytes(129, 300, 256) >= 256 * 256 * 4 + 256 * 4 + 300 * 4
    assert lq.lq_gemm_workspace_bytes(-1, 300, 256) == 0
    gm = lambda fmt=1, M=64, cols=2560, ws=FAKE, wsb=need, W=FAKE: L.lq_gemm(fmt, W, 128, cols, FAKE, FAKE, M, ws,
                                                                           wsb, None)
    assert gm(M=0) == lq.LQ_EINVAL
    assert gm(fmt=7) == lq.LQ_EINVAL
    assert gm(cols=2500) == lq.LQ_ESHAPE
    assert gm(wsb=need - 1) == lq.LQ_EWORKSPACE
    assert gm(ws=None) == lq.LQ_EWORKSPACE
    assert gm(ws=FAKE + 16) == lq.LQ_EALIGN


def test_gemm_gate_up_validation(lq):
    L = lq.lib()
    need = lq.lq_gemm_workspace_bytes(64, 256, 2560)
    gu = lambda fmt=1, inter=128, M=64, act=1, ws=FAKE, wsb=need: L.lq_gemm_gate_up_act(fmt, FAKE, inter, 2560, FAKE,
                                                                                        FAKE, M, act, ws, wsb, None)
    assert gu(act=0) == lq.LQ_EINVAL
    assert gu(act=3) == lq.LQ_EINVAL
    assert gu(M=0) == lq.LQ_EINVAL
    assert gu(fmt=7) == lq.LQ_EINVAL
    assert gu(inter=-1) == lq.LQ_ESHAPE
    assert gu(inter=0) == lq.LQ_OK
    assert gu(wsb=need - 1) == lq.LQ_EWORKSPACE
    assert gu(ws=FAKE + 16) == lq.LQ_EALIGN

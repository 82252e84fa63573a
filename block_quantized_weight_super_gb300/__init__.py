"""Python binding of liblq.so (include/lq.h): argument marshalling only.

Every function has the name of its C entry point and takes torch tensors
(device memory), plain ints for pointers, or None; `stream` is a
torch.cuda.Stream, a raw cudaStream_t int, or None for the current torch
stream.  A nonzero lq_status raises LqError.  There is no fallback: if the
library is not built, importing works but the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os

from . import build as _build

LIB_PATH = _build.LIB

LQ_Q4_K, LQ_Q6_K, LQ_Q8_0 = 1, 2, 3
LQ_ACT_GEGLU_TANH, LQ_ACT_SWIGLU = 1, 2
(LQ_OK, LQ_EINVAL, LQ_EALIGN, LQ_ESHAPE, LQ_EWORKSPACE, LQ_ECUDA, LQ_ETIMEOUT,
 LQ_EUNSUPPORTED) = range(8)

EXPORTS = ["lq_block_bytes", "lq_block_elems", "lq_row_bytes", "lq_status_str", "lq_last_error",
           "lq_dequant", "lq_matvec", "lq_matvec_softcap", "lq_matvec_act", "lq_gemm_workspace_bytes", "lq_gemm", "lq_gemm_gate_up_act", "lq_gemv_f16", "lq_gemv_f32", "lq_rmsnorm", "lq_qkv_mixed",
           "lq_qkv_mixed_rmsnorm", "lq_pack_gate_up", "lq_ffn_gate_up_act", "lq_ffn_gate_up_act_rmsnorm",
           "lq_ffn", "lq_moe_workspace_bytes", "lq_moe_ffn", "lq_moe_ffn_ex_workspace_bytes", "lq_moe_ffn_ex",
           "lq_moe_ffn_static",
           "lq_device_status",
           "lq_set_wait_timeout_ns", "lq_probe_timeout"]

LQ_MOE_STATIC_SCRATCH_BYTES = 4 << 20
LQ_MOE_MAX_SHARED = 16
LQ_GEMM_MIN_M = 32


class LqError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


_lib = None


def lib():
    """load liblq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        i32, i64, vp, sz, u64 = C.c_int, C.c_int64, C.c_void_p, C.c_size_t, C.c_uint64
        sig = {
            "lq_block_bytes": ([i32], sz),
            "lq_block_elems": ([i32], i32),
            "lq_row_bytes": ([i32, i64], i64),
            "lq_status_str": ([i32], C.c_char_p),
            "lq_last_error": ([], C.c_char_p),
            "lq_dequant": ([i32, vp, i64, i64, vp, vp], i32),
            "lq_matvec": ([i32, vp, i64, i64, vp, vp, i32, vp], i32),
            "lq_matvec_softcap": ([i32, vp, i64, i64, vp, vp, i32, C.c_float, vp], i32),
            "lq_matvec_act": ([i32, vp, i64, i64, vp, vp, vp, i32, i32, vp], i32),
            "lq_gemm_workspace_bytes": ([i64, i64, i64], sz),
            "lq_gemm": ([i32, vp, i64, i64, vp, vp, i64, vp, sz, vp], i32),
            "lq_gemm_gate_up_act": ([i32, vp, i64, i64, vp, vp, i64, i32, vp, sz, vp], i32),
            "lq_gemv_f16": ([vp, i64, i64, vp, vp, i32, vp], i32),
            "lq_gemv_f32": ([vp, i64, i64, vp, vp, i32, vp], i32),
            "lq_rmsnorm": ([vp, vp, C.c_float, vp, i32, i64, vp], i32),
            "lq_qkv_mixed": ([i32, vp, i64, i32, vp, i64, i32, vp, i64, i64, vp, vp, vp, vp, i32, vp], i32),
            "lq_qkv_mixed_rmsnorm": ([i32, vp, i64, i32, vp, i64, i32, vp, i64, i64, vp, vp, C.c_float, vp, vp, vp,
                                      vp, i32, vp], i32),
            "lq_ffn_gate_up_act_rmsnorm": ([i32, vp, i64, i64, vp, vp, C.c_float, vp, vp, i32, i32, vp], i32),
            "lq_pack_gate_up": ([i32, vp, vp, i64, i64, vp, vp], i32),
            "lq_ffn_gate_up_act": ([i32, vp, i64, i64, vp, vp, i32, i32, vp], i32),
            "lq_ffn": ([i32, vp, i32, vp, i64, i64, vp, vp, vp, i32, i32, vp], i32),
            "lq_moe_workspace_bytes": ([i32, i32, i32, i64, i64], sz),
            "lq_moe_ffn": ([vp, i32, i32, i32, vp, vp, vp, i64, i64, vp, vp, i32, vp, vp, vp, sz, vp], i32),
            "lq_moe_ffn_ex_workspace_bytes": ([i32, i32, i32, i64, i64, i32, i64], sz),
            "lq_moe_ffn_ex": ([vp, i32, i32, i32, i32, vp, vp, vp, i64, i64, i32, vp, vp, vp, i64, vp, vp, vp, i32,
                               vp, vp, vp, sz, vp], i32),
            "lq_moe_ffn_static": ([vp, i32, i32, i32, vp, vp, vp, i64, i64, vp, vp, i32, vp, vp, vp], i32),
            "lq_device_status": ([vp, C.POINTER(C.c_uint32)], i32),
            "lq_set_wait_timeout_ns": ([u64], None),
            "lq_probe_timeout": ([u64, vp], i32),
        }
        for name, (args, res) in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(rc: int):
    if rc != LQ_OK:
        raise LqError(rc, lib().lq_last_error().decode() or lib().lq_status_str(rc).decode())
    return rc


def lq_block_bytes(fmt: int) -> int:
    return lib().lq_block_bytes(fmt)


def lq_block_elems(fmt: int) -> int:
    return lib().lq_block_elems(fmt)


def lq_row_bytes(fmt: int, cols: int) -> int:
    return lib().lq_row_bytes(fmt, cols)


def lq_status_str(status: int) -> str:
    return lib().lq_status_str(status).decode()


def lq_last_error() -> str:
    return lib().lq_last_error().decode()


def lq_dequant(fmt, W, rows, cols, out, stream=None):
    return _check(lib().lq_dequant(fmt, _ptr(W), rows, cols, _ptr(out), _stream(stream)))


def lq_matvec(fmt, W, rows, cols, x, y, batch, stream=None):
    return _check(lib().lq_matvec(fmt, _ptr(W), rows, cols, _ptr(x), _ptr(y), batch, _stream(stream)))


def lq_matvec_softcap(fmt, W, rows, cols, x, y, batch, cap, stream=None):
    return _check(lib().lq_matvec_softcap(fmt, _ptr(W), rows, cols, _ptr(x), _ptr(y), batch, float(cap),
                                          _stream(stream)))


def lq_matvec_act(fmt, W, rows, cols, gu, h, y, batch, act, stream=None):
    return _check(lib().lq_matvec_act(fmt, _ptr(W), rows, cols, _ptr(gu), _ptr(h), _ptr(y), batch, act,
                                      _stream(stream)))


def lq_gemm_workspace_bytes(M, rows, cols) -> int:
    return lib().lq_gemm_workspace_bytes(M, rows, cols)


def lq_gemm(fmt, W, rows, cols, X, Y, M, workspace=None, ws_bytes=0, stream=None):
    return _check(lib().lq_gemm(fmt, _ptr(W), rows, cols, _ptr(X), _ptr(Y), M, _ptr(workspace), ws_bytes,
                                _stream(stream)))


def lq_gemm_gate_up_act(fmt, Wgu, inter, cols, X, H, M, act, workspace=None, ws_bytes=0, stream=None):
    return _check(lib().lq_gemm_gate_up_act(fmt, _ptr(Wgu), inter, cols, _ptr(X), _ptr(H), M, act, _ptr(workspace),
                                            ws_bytes, _stream(stream)))


def lq_gemv_f16(W, rows, cols, x, y, batch, stream=None):
    return _check(lib().lq_gemv_f16(_ptr(W), rows, cols, _ptr(x), _ptr(y), batch, _stream(stream)))


def lq_gemv_f32(W, rows, cols, x, y, batch, stream=None):
    return _check(lib().lq_gemv_f32(_ptr(W), rows, cols, _ptr(x), _ptr(y), batch, _stream(stream)))


def lq_rmsnorm(x, w, eps, out, ntok, n, stream=None):
    return _check(lib().lq_rmsnorm(_ptr(x), _ptr(w), float(eps), _ptr(out), ntok, n, _stream(stream)))


def lq_qkv_mixed_rmsnorm(fq, Wq, nq, fk, Wk, nk, fv, Wv, nv, cols, x, norm_w, eps, xn, q, k, v, batch,
                         stream=None):
    return _check(lib().lq_qkv_mixed_rmsnorm(fq, _ptr(Wq), nq, fk, _ptr(Wk), nk, fv, _ptr(Wv), nv, cols, _ptr(x),
                                             _ptr(norm_w), float(eps), _ptr(xn), _ptr(q), _ptr(k), _ptr(v), batch,
                                             _stream(stream)))


def lq_ffn_gate_up_act_rmsnorm(fmt, Wgu, inter, cols, x, norm_w, eps, xn, h, batch, act, stream=None):
    return _check(lib().lq_ffn_gate_up_act_rmsnorm(fmt, _ptr(Wgu), inter, cols, _ptr(x), _ptr(norm_w), float(eps),
                                                   _ptr(xn), _ptr(h), batch, act, _stream(stream)))


def lq_qkv_mixed(fq, Wq, nq, fk, Wk, nk, fv, Wv, nv, cols, x, q, k, v, batch, stream=None):
    return _check(lib().lq_qkv_mixed(fq, _ptr(Wq), nq, fk, _ptr(Wk), nk, fv, _ptr(Wv), nv, cols,
                                     _ptr(x), _ptr(q), _ptr(k), _ptr(v), batch, _stream(stream)))


def lq_pack_gate_up(fmt, Wg, Wu, inter, cols, Wgu_out, stream=None):
    return _check(lib().lq_pack_gate_up(fmt, _ptr(Wg), _ptr(Wu), inter, cols, _ptr(Wgu_out),
                                        _stream(stream)))


def lq_ffn_gate_up_act(fmt, Wgu, inter, cols, x, h, batch, act, stream=None):
    return _check(lib().lq_ffn_gate_up_act(fmt, _ptr(Wgu), inter, cols, _ptr(x), _ptr(h), batch,
                                           act, _stream(stream)))


def lq_ffn(fmt_gu, Wgu, fmt_down, Wd, inter, hidden, x, h, y, batch, act, stream=None):
    return _check(lib().lq_ffn(fmt_gu, _ptr(Wgu), fmt_down, _ptr(Wd), inter, hidden, _ptr(x), _ptr(h),
                               _ptr(y), batch, act, _stream(stream)))


def lq_moe_workspace_bytes(n_experts, topk, ntok, hidden, inter) -> int:
    return lib().lq_moe_workspace_bytes(n_experts, topk, ntok, hidden, inter)


def _ptr_array(ts):
    arr = (C.c_void_p * len(ts))(*[_ptr(t) for t in ts])
    return arr


def lq_moe_ffn(router, n_experts, topk, fmt, W1, W3, W2, hidden, inter, X, Y, ntok,
               topk_idx=None, topk_w=None, workspace=None, ws_bytes=0, stream=None):
    a1, a3, a2 = _ptr_array(W1), _ptr_array(W3), _ptr_array(W2)
    return _check(lib().lq_moe_ffn(_ptr(router), n_experts, topk, fmt, C.cast(a1, C.c_void_p),
                                   C.cast(a3, C.c_void_p), C.cast(a2, C.c_void_p), hidden, inter,
                                   _ptr(X), _ptr(Y), ntok, _ptr(topk_idx), _ptr(topk_w),
                                   _ptr(workspace), ws_bytes, _stream(stream)))


def lq_moe_ffn_ex_workspace_bytes(n_experts, topk, ntok, hidden, inter, n_shared, inter_s) -> int:
    return lib().lq_moe_ffn_ex_workspace_bytes(n_experts, topk, ntok, hidden, inter, n_shared, inter_s)


def lq_moe_ffn_ex(router, n_experts, topk, norm_topk_prob, fmt, W1, W3, W2, hidden, inter, X, Y, ntok,
                  Ws1=(), Ws3=(), Ws2=(), inter_s=0, shared_gate=None, topk_idx=None, topk_w=None,
                  workspace=None, ws_bytes=0, stream=None):
    a1, a3, a2 = _ptr_array(W1), _ptr_array(W3), _ptr_array(W2)
    ns = len(Ws1)
    s1, s3, s2 = (_ptr_array(Ws1), _ptr_array(Ws3), _ptr_array(Ws2)) if ns else (None, None, None)
    cast = lambda a: None if a is None else C.cast(a, C.c_void_p)
    return _check(lib().lq_moe_ffn_ex(_ptr(router), n_experts, topk, norm_topk_prob, fmt, cast(a1), cast(a3),
                                      cast(a2), hidden, inter, ns, cast(s1), cast(s3), cast(s2), inter_s,
                                      _ptr(shared_gate), _ptr(X), _ptr(Y), ntok, _ptr(topk_idx), _ptr(topk_w),
                                      _ptr(workspace), ws_bytes, _stream(stream)))


def lq_moe_ffn_static(router, n_experts, topk, fmt, W1, W3, W2, hidden, inter, X, Y, ntok,
                      topk_idx=None, topk_w=None, stream=None):
    a1, a3, a2 = _ptr_array(W1), _ptr_array(W3), _ptr_array(W2)
    return _check(lib().lq_moe_ffn_static(_ptr(router), n_experts, topk, fmt, C.cast(a1, C.c_void_p),
                                          C.cast(a3, C.c_void_p), C.cast(a2, C.c_void_p), hidden, inter,
                                          _ptr(X), _ptr(Y), ntok, _ptr(topk_idx), _ptr(topk_w),
                                          _stream(stream)))


def lq_device_status(stream=None):
    """returns (status code, bits) without raising."""
    bits = C.c_uint32(0)
    rc = lib().lq_device_status(_stream(stream), C.byref(bits))
    return rc, bits.value


def lq_set_wait_timeout_ns(ns: int):
    lib().lq_set_wait_timeout_ns(ns)


def lq_probe_timeout(timeout_ns, stream=None):
    return _check(lib().lq_probe_timeout(timeout_ns, _stream(stream)))

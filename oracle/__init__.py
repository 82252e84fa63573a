"""CPU oracle for the block-quantized decode matvec -- TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 C++ (``lq_oracle.cpp``) behind a numpy/ctypes wrapper.  It
shares no code with the CUDA library and the library never imports it; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it.

What it computes, and the passages it follows, is stated at the top of
``lq_oracle.cpp``.  ``build()`` compiles it with g++ (no GPU needed).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "lq_oracle.cpp")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "liblq_oracle.so")

Q4_K, Q6_K, Q8_0 = 1, 2, 3
ACT_GEGLU_TANH, ACT_SWIGLU = 1, 2

_lib = None


def build(force: bool = False) -> str:
    """compile the oracle to a shared library (g++, -ffp-contract=off)."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(LIB)
        i64, i32, vp, d = C.c_int64, C.c_int, C.c_void_p, C.c_double
        L.orc_block_bytes.argtypes = [i32]
        L.orc_block_elems.argtypes = [i32]
        L.orc_half_to_double.argtypes = [C.c_uint16]
        L.orc_half_to_double.restype = d
        L.orc_gelu_tanh.argtypes = [d]
        L.orc_gelu_tanh.restype = d
        L.orc_silu.argtypes = [d]
        L.orc_silu.restype = d
        L.orc_softcap.argtypes = [vp, i64, d, vp]
        L.orc_softcap.restype = None
        L.orc_rmsnorm.argtypes = [vp, i32, i64, vp, d, vp]
        L.orc_rmsnorm.restype = None
        L.orc_moe_weights_raw.argtypes = [vp, i32, i32, vp, i32, vp]
        L.orc_moe_weights_raw.restype = None
        L.orc_moe_shared.argtypes = [i32, vp, vp, vp, i32, i64, i64, vp, i32, vp, vp, vp, i32]
        L.orc_moe_shared.restype = None
        L.orc_dequant.argtypes = [i32, vp, i64, i64, vp, i32]
        L.orc_matvec.argtypes = [i32, vp, i64, i64, vp, i32, vp, vp, i32]
        L.orc_matvec_rows.argtypes = [i32, vp, i64, vp, i64, vp, i32, vp, vp, i32]
        L.orc_ffn_gate_up.argtypes = [i32, vp, vp, i64, i64, vp, i32, i32, vp, vp, vp, vp, vp, i32]
        L.orc_moe_route.argtypes = [vp, i32, i64, vp, i32, i32, vp, vp, vp, vp]
        L.orc_moe_ffn.argtypes = [i32, vp, vp, vp, i64, i64, vp, i32, i32, vp, vp, vp, vp, vp,
                                  vp, vp, vp, vp, vp, i32]
        L.orc_abs_matvec.argtypes = [i32, vp, i64, i64, vp, vp, i32]
        L.orc_moe_weights.argtypes = [vp, i32, i32, vp, i32, vp]
        _lib = L
    return _lib


def _u8(W):
    W = np.ascontiguousarray(W)
    assert W.dtype == np.uint8
    return W


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def threads_default() -> int:
    return os.cpu_count() or 1


def block_bytes(fmt: int) -> int:
    return lib().orc_block_bytes(fmt)


def block_elems(fmt: int) -> int:
    return lib().orc_block_elems(fmt)


def half_to_double(bits: int) -> float:
    return lib().orc_half_to_double(bits)


def gelu_tanh(g: float) -> float:
    return lib().orc_gelu_tanh(g)


def silu(g: float) -> float:
    return lib().orc_silu(g)


def rmsnorm(X, w, eps: float) -> np.ndarray:
    """RMS-norm of each row of X [ntok][n] with weight w [n]: x * w / sqrt(mean(x^2) + eps), fp64."""
    X = _f32(X)
    X2 = X.reshape(-1, X.shape[-1])
    w = _f32(w)
    out = np.empty(X2.shape, dtype=np.float64)
    lib().orc_rmsnorm(_p(X2), X2.shape[0], X2.shape[1], _p(w), float(eps), _p(out))
    return out.reshape(X.shape)


def softcap(y, cap: float) -> np.ndarray:
    """final-logit soft-cap cap * tanh(y / cap), elementwise, fp64."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    out = np.empty_like(y)
    lib().orc_softcap(_p(y), y.size, float(cap), _p(out))
    return out


def dequant(fmt: int, W, rows: int, cols: int, nthreads: int = 1) -> np.ndarray:
    W = _u8(W)
    out = np.empty((rows, cols), dtype=np.float32)
    lib().orc_dequant(fmt, _p(W), rows, cols, _p(out), nthreads)
    return out


def matvec(fmt: int, W, rows: int, cols: int, x, nthreads: int = 1):
    """y = dequant(W) . x for x [batch][cols]; returns (y, S) each [batch][rows] fp64."""
    W, x = _u8(W), _f32(x)
    x2 = x.reshape(-1, cols)
    batch = x2.shape[0]
    y = np.empty((batch, rows), dtype=np.float64)
    S = np.empty((batch, rows), dtype=np.float64)
    lib().orc_matvec(fmt, _p(W), rows, cols, _p(x2), batch, _p(y), _p(S), nthreads)
    return y, S


def matvec_rows(fmt: int, W, cols: int, row_idx, x, nthreads: int = 1):
    W, x = _u8(W), _f32(x)
    idx = np.ascontiguousarray(row_idx, dtype=np.int64)
    x2 = x.reshape(-1, cols)
    batch = x2.shape[0]
    y = np.empty((batch, idx.size), dtype=np.float64)
    S = np.empty((batch, idx.size), dtype=np.float64)
    lib().orc_matvec_rows(fmt, _p(W), cols, _p(idx), idx.size, _p(x2), batch, _p(y), _p(S),
                          nthreads)
    return y, S


def ffn_gate_up(fmt: int, Wg, Wu, inter: int, cols: int, x, act: int, nthreads: int = 1):
    """returns dict of fp64 [batch][inter] arrays: h, g, u, Sg, Su."""
    Wg, Wu, x = _u8(Wg), _u8(Wu), _f32(x)
    x2 = x.reshape(-1, cols)
    batch = x2.shape[0]
    out = {k: np.empty((batch, inter), dtype=np.float64) for k in ("h", "g", "u", "Sg", "Su")}
    lib().orc_ffn_gate_up(fmt, _p(Wg), _p(Wu), inter, cols, _p(x2), batch, act, _p(out["h"]),
                          _p(out["g"]), _p(out["u"]), _p(out["Sg"]), _p(out["Su"]), nthreads)
    return out


def moe_route(R, X, topk: int):
    R, X = _f32(R), _f32(X)
    E, hidden = R.shape
    ntok = X.shape[0]
    idx = np.empty((ntok, topk), dtype=np.int32)
    w = np.empty((ntok, topk), dtype=np.float64)
    logits = np.empty((ntok, E), dtype=np.float64)
    labs = np.empty((ntok, E), dtype=np.float64)
    lib().orc_moe_route(_p(R), E, hidden, _p(X), ntok, topk, _p(idx), _p(w), _p(logits),
                        _p(labs))
    return idx, w, logits, labs


def moe_weights(logits, idx, norm: bool = True):
    """routing weights of a given selection idx [ntok][topk] from fp64 logits
    [ntok][E]: the selected softmax probabilities, renormalised by their sum
    (norm) or as they are (norm_topk_prob = false)."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    ntok, E = logits.shape
    w = np.empty(idx.shape, dtype=np.float64)
    f = lib().orc_moe_weights if norm else lib().orc_moe_weights_raw
    f(_p(logits), E, ntok, _p(idx), idx.shape[1], _p(w))
    return w


def moe_shared(fmt: int, Wg, Wu, Wd, hidden: int, inter_s: int, X, gate=None, nthreads: int = 1):
    """shared-expert branch: gate_t * sum_s Wd_s (silu(Wg_s x_t) * (Wu_s x_t)),
    gate_t = sigmoid(g . x_t) (or 1 without g).  Returns (S [ntok][hidden],
    gate_t [ntok]), fp64."""
    Wg, Wu, Wd = [_u8(a) for a in Wg], [_u8(a) for a in Wu], [_u8(a) for a in Wd]
    n = len(Wg)
    P = C.c_void_p * n
    pg, pu, pd = P(*[_p(a) for a in Wg]), P(*[_p(a) for a in Wu]), P(*[_p(a) for a in Wd])
    X = _f32(X)
    ntok = X.shape[0]
    g = None if gate is None else _f32(gate)
    S = np.empty((ntok, hidden))
    gs = np.empty(ntok)
    lib().orc_moe_shared(fmt, C.cast(pg, C.c_void_p), C.cast(pu, C.c_void_p), C.cast(pd, C.c_void_p), n,
                         hidden, inter_s, _p(X), ntok, None if g is None else _p(g), _p(S), _p(gs), nthreads)
    return S, gs


def moe_ffn(fmt: int, W1, W3, W2, hidden: int, inter: int, X, idx, w, nthreads: int = 1):
    """expert FFN + weighted combine for a given routing (idx, w)."""
    W1 = [_u8(a) for a in W1]
    W3 = [_u8(a) for a in W3]
    W2 = [_u8(a) for a in W2]
    E = len(W1)
    P = C.c_void_p * E
    p1, p3, p2 = P(*[_p(a) for a in W1]), P(*[_p(a) for a in W3]), P(*[_p(a) for a in W2])
    X = _f32(X)
    ntok = X.shape[0]
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    topk = idx.shape[1]
    w = np.ascontiguousarray(w, dtype=np.float64)
    nslot = ntok * topk
    out = {
        "Y": np.empty((ntok, hidden)),
        "ye": np.empty((nslot, hidden)),
        "Sy": np.empty((nslot, hidden)),
        "h": np.empty((nslot, inter)),
        "g": np.empty((nslot, inter)),
        "u": np.empty((nslot, inter)),
        "Sg": np.empty((nslot, inter)),
        "Su": np.empty((nslot, inter)),
    }
    lib().orc_moe_ffn(fmt, C.cast(p1, C.c_void_p), C.cast(p3, C.c_void_p),
                      C.cast(p2, C.c_void_p), hidden, inter, _p(X), ntok, topk, _p(idx), _p(w),
                      _p(out["Y"]), _p(out["ye"]), _p(out["Sy"]), _p(out["h"]), _p(out["g"]),
                      _p(out["u"]), _p(out["Sg"]), _p(out["Su"]), nthreads)
    return out


def dense_matvec(W, x):
    """y = W . x for a non-quantized W (fp16 or fp32 [rows][cols], each value
    taken exactly in fp64) and x [batch][cols] fp32; returns (y, S) with
    S = sum_j |w_ij x_j|, both [batch][rows] fp64 (larql Gemma 3 table,
    lm_head row: the f16_gemv / f32_gemv fallbacks).  A library matmul in
    fp64 is the step: every product of two fp16/fp32 values is exact in
    fp64, and its sums carry ~1e-16 relative error."""
    W64 = np.asarray(W).astype(np.float64)
    x64 = np.atleast_2d(np.asarray(x, dtype=np.float32)).astype(np.float64)
    return x64 @ W64.T, np.abs(x64) @ np.abs(W64).T


def abs_matvec(fmt: int, W, rows: int, cols: int, v, nthreads: int = 1) -> np.ndarray:
    """sum_j |w_ij| v_j for each row (carries an input bound through a matvec)."""
    W = _u8(W)
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(rows, dtype=np.float64)
    lib().orc_abs_matvec(fmt, _p(W), rows, cols, _p(v), _p(out), nthreads)
    return out


# ---------------------------------------------------------------------------
# Error bounds the GPU results are held to (functions of oracle quantities).
# ---------------------------------------------------------------------------
U32 = 2.0 ** -24


def matvec_bound(S):
    """|y_gpu - y| <= 1e-5 * sum_j |w_ij x_j| + 1e-6 per element."""
    return 1e-5 * np.asarray(S) + 1e-6


def softcap_bound(S, y, cap: float):
    """bound on a soft-capped output whose pre-cap value carries the matvec
    bound: the map has slope at most 1, so that bound carries over; fp32
    evaluation adds the rounding of y / cap (slope <= 1: u32 |y|), tanhf
    (2 ulps of the result) and the final product (1 ulp): 8 u32 (|y| + cap)
    covers them with room."""
    return matvec_bound(S) + 8 * U32 * (np.abs(np.asarray(y, dtype=np.float64)) + cap)


def act_abs(g, act: int):
    g = np.asarray(g, dtype=np.float64)
    if act == ACT_GEGLU_TANH:
        k = np.sqrt(2.0 / np.pi)
        a = 0.5 * g * (1.0 + np.tanh(k * (g + 0.044715 * g ** 3)))
    else:
        a = g / (1.0 + np.exp(-g))
    return np.abs(a)


def gate_up_bound(g, u, Sg, Su, act: int):
    """per-element bound on h = act(g)*u when g and u each carry the matvec
    bound: 1.2 e_g (|u| + e_u) + |act(g)| e_u + 8 u32 (|act(g)| + 1.2 e_g)(|u| + e_u).

    1.2 bounds |act'| for both GELU-tanh and SiLU; the last term covers the
    fp32 evaluation of the activation and of the product."""
    eg, eu = matvec_bound(Sg), matvec_bound(Su)
    a = act_abs(g, act)
    au = np.abs(u) + eu
    return 1.2 * eg * au + a * eu + 8 * U32 * (a + 1.2 * eg) * au


def moe_check(fmt: int, W1, W3, W2, hidden: int, inter: int, X, logits, labs, idx_gpu,
              nthreads: int = 1, norm: bool = True):
    """Oracle result and per-element bound for the MoE evaluated on the GPU's
    expert selection idx_gpu [ntok][topk].

    Returns dict: Y (fp64 reference), bound, w (oracle weights of the selection),
    admissible (bool per token: the selection is a valid top-k within the
    logits' error e_l = 1e-5*sum|R x| + 1e-6).
    Bound per output: sum_k w_k B_y,k + |y_k| (2 w_k e_lmax + 8 u32 w_k), with
    B_y = 1e-5 Sy + 1e-6 + sum_j |w2_ij| B_h,j and B_h the gate/up bound.
    norm: renormalised weights (True) or the raw selected softmax
    probabilities (False); either way log w_k moves by at most 2 e_lmax when
    the logits move by e_l (|d log p_k| <= |d l_k| + max |d l|), so the
    same bound holds."""
    idx_gpu = np.ascontiguousarray(idx_gpu, dtype=np.int32)
    ntok, topk = idx_gpu.shape
    E = logits.shape[1]
    el = 1e-5 * np.asarray(labs) + 1e-6
    adm = np.zeros(ntok, dtype=bool)
    for t in range(ntok):
        sel = set(int(e) for e in idx_gpu[t])
        if len(sel) != topk or min(sel) < 0 or max(sel) >= E:
            continue
        rest = [e for e in range(E) if e not in sel]
        ok = all(logits[t, a] + el[t, a] >= logits[t, b] - el[t, b] for a in sel for b in rest)
        adm[t] = ok
    w = moe_weights(logits, idx_gpu, norm)
    out = moe_ffn(fmt, W1, W3, W2, hidden, inter, X, idx_gpu, w, nthreads)
    Bh = gate_up_bound(out["g"], out["u"], out["Sg"], out["Su"], ACT_SWIGLU)
    bound = np.zeros((ntok, hidden))
    for t in range(ntok):
        elmax = el[t].max()
        for k in range(topk):
            s = t * topk + k
            e = int(idx_gpu[t, k])
            By = 1e-5 * out["Sy"][s] + 1e-6 + abs_matvec(fmt, W2[e], hidden, inter, Bh[s], nthreads)
            bound[t] += w[t, k] * By + np.abs(out["ye"][s]) * (2 * w[t, k] * elmax + 8 * U32 * w[t, k])
    return {"Y": out["Y"], "bound": bound, "w": w, "admissible": adm, "el": el, "ye": out["ye"]}

"""Pins of the oracle's matvec, gated-FFN and MoE arithmetic against facts
outside it: one-hot and all-ones inputs, numpy/torch library routines on tiny
cases, linearity, closed forms of the routing rule, and the dotLLM MoE unit
tests (tie stability, one-hot router, uniform router, scalar reference)."""
import math

import numpy as np
import pytest
import torch

import synth
from blockpack import pack_q4k
from conftest import golden_lines

Q4_K, Q6_K, Q8_0 = 1, 2, 3
FMTS = [Q4_K, Q6_K, Q8_0]


def _mat(fmt, rows, cols, seed=0):
    g = synth.rng(seed)
    return synth.weights(g, fmt, rows, cols), synth.activations(g, 3, cols)


@pytest.mark.parametrize("fmt", FMTS)
def test_one_hot_x_gives_dequant_column(orc, fmt):
    rows, cols = 5, 2 * orc.block_elems(fmt) * 2
    W, _ = _mat(fmt, rows, cols)
    D = orc.dequant(fmt, W, rows, cols)
    for j in [0, 1, 31, 32, cols // 2 + 3, cols - 1]:
        x = np.zeros((1, cols), dtype=np.float32)
        x[0, j] = 1.0
        y, S = orc.matvec(fmt, W, rows, cols, x)
        assert np.array_equal(y[0], D[:, j].astype(np.float64))
        assert np.array_equal(S[0], np.abs(D[:, j]).astype(np.float64))


@pytest.mark.parametrize("fmt", FMTS)
def test_all_ones_gives_row_sums(orc, fmt):
    rows, cols = 7, orc.block_elems(fmt) * 4
    W, _ = _mat(fmt, rows, cols, seed=1)
    D = orc.dequant(fmt, W, rows, cols).astype(np.float64)
    y, _ = orc.matvec(fmt, W, rows, cols, np.ones((1, cols), dtype=np.float32))
    assert np.allclose(y[0], D.sum(axis=1), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("fmt", FMTS)
def test_tiny_brute_force_vs_numpy(orc, fmt):
    """rows <= 4, one super-block: against numpy's fp64 matmul of the dequantized W."""
    for rows in (1, 2, 3, 4):
        cols = orc.block_elems(fmt)
        W, X = _mat(fmt, rows, cols, seed=rows)
        D = orc.dequant(fmt, W, rows, cols).astype(np.float64)
        y, S = orc.matvec(fmt, W, rows, cols, X)
        ref = X.astype(np.float64) @ D.T
        assert np.allclose(y, ref, rtol=1e-13, atol=1e-14)
        assert np.allclose(S, np.abs(X.astype(np.float64)) @ np.abs(D.T), rtol=1e-13)


def test_tiny_hand_expansion(orc):
    """a hand-expanded 1 x 256 Q4_K row: w = d*sc_j*q - dmin*m_j by sub-block."""
    sc = [1, 2, 3, 4, 5, 6, 7, 8]
    m = [0, 1, 0, 1, 0, 1, 0, 1]
    q = np.tile(np.arange(16), 16)
    blk = pack_q4k(0.5, 0.25, sc, m, q).reshape(1, -1)
    x = np.linspace(-1, 1, 256, dtype=np.float32).reshape(1, -1)
    expect = 0.0
    for i in range(256):
        j = i // 32
        expect += (0.5 * sc[j] * q[i] - 0.25 * m[j]) * float(x[0, i])
    y, _ = orc.matvec(Q4_K, blk, 1, 256, x)
    assert abs(y[0, 0] - expect) <= 1e-12 * abs(expect) + 1e-15


@pytest.mark.parametrize("fmt", FMTS)
def test_linearity(orc, fmt):
    rows, cols = 6, orc.block_elems(fmt) * 3
    W, X = _mat(fmt, rows, cols, seed=9)
    a, b = 2.0, -0.5        # powers of two on disjoint supports: a*x + b*x' exact in fp32
    half = cols // 2
    xa, xb = X[0:1].copy(), X[1:2].copy()
    xa[:, half:] = 0
    xb[:, :half] = 0
    comb = (np.float32(a) * xa + np.float32(b) * xb).astype(np.float32)
    assert np.array_equal(comb.astype(np.float64), a * xa.astype(np.float64) + b * xb.astype(np.float64))
    y1, S1 = orc.matvec(fmt, W, rows, cols, xa)
    y2, S2 = orc.matvec(fmt, W, rows, cols, xb)
    y3, _ = orc.matvec(fmt, W, rows, cols, comb)
    assert np.allclose(y3, a * y1 + b * y2, rtol=0, atol=1e-12 * (S1 + S2).max())


@pytest.mark.parametrize("fmt", FMTS)
def test_batch_rows_independent(orc, fmt):
    rows, cols = 4, orc.block_elems(fmt) * 2
    W, X = _mat(fmt, rows, cols, seed=10)
    Y, S = orc.matvec(fmt, W, rows, cols, X)
    for b in range(X.shape[0]):
        yb, Sb = orc.matvec(fmt, W, rows, cols, X[b:b + 1])
        assert np.array_equal(Y[b], yb[0]) and np.array_equal(S[b], Sb[0])


def test_q8_0_row_stride_regression_shapes(orc):
    """rows of an odd number of 34-byte blocks: each row equals that row on its own."""
    for line in golden_lines("q8_0_stride_shapes.txt"):
        M, K = map(int, line.split())
        W, X = _mat(Q8_0, M, K, seed=M * 1000 + K)
        y, _ = orc.matvec(Q8_0, W, M, K, X[:1])
        for r in range(M):
            yr, _ = orc.matvec(Q8_0, W[r:r + 1], 1, K, X[:1])
            assert y[0, r] == yr[0, 0]


@pytest.mark.parametrize("fmt", FMTS)
def test_matvec_rows_and_threads(orc, fmt):
    rows, cols = 37, orc.block_elems(fmt) * 3
    W, X = _mat(fmt, rows, cols, seed=11)
    y, S = orc.matvec(fmt, W, rows, cols, X)
    y4, S4 = orc.matvec(fmt, W, rows, cols, X, nthreads=4)
    assert np.array_equal(y, y4) and np.array_equal(S, S4)
    idx = np.array([36, 0, 5, 5, 17])
    yr, Sr = orc.matvec_rows(fmt, W, cols, idx, X, nthreads=3)
    assert np.array_equal(yr, y[:, idx]) and np.array_equal(Sr, S[:, idx])


# ---------------------------------------------------------------- activations

def test_gelu_tanh_vs_torch(orc):
    g = np.concatenate([np.linspace(-12, 12, 4001), [0.0, 1e-8, -1e-8, 30.0, -30.0]])
    got = np.array([orc.gelu_tanh(v) for v in g])
    ref = torch.nn.functional.gelu(torch.tensor(g, dtype=torch.float64), approximate="tanh").numpy()
    # 1 + tanh(z) cancels for very negative g: absolute error ~ |g| * 2^-53
    tol = 1e-13 * np.abs(ref) + 4e-16 * np.abs(g)
    assert np.all(np.abs(got - ref) <= tol)
    # independent closed form: 0.5 (1 + tanh z) = 1 / (1 + exp(-2 z))
    z = math.sqrt(2 / math.pi) * (g + 0.044715 * g ** 3)
    alt = g / (1 + np.exp(-2 * z))
    assert np.all(np.abs(got - alt) <= 1e-13 * np.abs(alt) + 4e-16 * np.abs(g))
    assert orc.gelu_tanh(0.0) == 0.0
    assert abs(orc.gelu_tanh(30.0) - 30.0) < 1e-12


def test_silu_vs_torch(orc):
    g = np.linspace(-40, 40, 4001)
    got = np.array([orc.silu(v) for v in g])
    ref = torch.nn.functional.silu(torch.tensor(g, dtype=torch.float64)).numpy()
    assert np.allclose(got, ref, rtol=1e-14, atol=1e-300)
    assert orc.silu(0.0) == 0.0


@pytest.mark.parametrize("act", [1, 2])
def test_activation_slope_below_bound(orc, act):
    """|act'| < 1.2 everywhere, the constant the post-activation bound uses."""
    f = orc.gelu_tanh if act == 1 else orc.silu
    g = np.linspace(-20, 20, 40001)
    v = np.array([f(t) for t in g])
    assert np.abs(np.diff(v) / np.diff(g)).max() < 1.2


# ---------------------------------------------------------------- final-logit soft-cap

@pytest.mark.parametrize("cap", [30.0, 50.0, 0.5])
def test_softcap_pins(orc, cap):
    """cap * tanh(y / cap) against facts outside the formula: zero, odd
    symmetry, its third-order series, the inverse through the library's
    atanh, saturation, monotonicity, and the (-cap, cap) band that the dotLLM
    FinalLogitSoftcap test asserts."""
    assert orc.softcap(np.array([0.0]), cap)[0] == 0.0
    y = np.linspace(-20 * cap, 20 * cap, 8001)
    out = orc.softcap(y, cap)
    assert np.array_equal(orc.softcap(-y, cap), -out)                    # odd
    assert np.all(np.abs(out) <= cap) and np.all(np.diff(out) >= 0)       # band, non-decreasing
    inner = np.abs(y[:-1]) <= 5 * cap                                   # tanh is not yet 1.0 in fp64
    assert np.all(np.diff(out)[inner] > 0)                              # strictly increasing there
    assert abs(out[-1] - cap) < 1e-12 * cap                              # saturation at 20 cap
    small = cap * np.array([1e-4, -3e-4, 1e-3])
    series = small - small ** 3 / (3 * cap ** 2)                        # tanh t = t - t^3/3 + O(t^5)
    assert np.all(np.abs(orc.softcap(small, cap) - series) <= 1e-12 * np.abs(small))
    t = np.array([0.1, 0.5, 0.9, -0.75])
    assert np.allclose(orc.softcap(cap * np.arctanh(t), cap), cap * t, rtol=1e-14, atol=0)   # inverse
    grad = np.diff(out) / np.diff(y)
    assert grad.max() <= 1.0 + 1e-9                                      # slope <= 1 (the bound uses it)


# ---------------------------------------------------------------- gated FFN

@pytest.mark.parametrize("act", [1, 2])
@pytest.mark.parametrize("fmt", [Q4_K, Q8_0])
def test_ffn_gate_up_composition(orc, fmt, act):
    inter, cols = 9, orc.block_elems(fmt) * 2
    g_ = synth.rng(12)
    Wg = synth.weights(g_, fmt, inter, cols)
    Wu = synth.weights(g_, fmt, inter, cols)
    X = synth.activations(g_, 2, cols)
    out = orc.ffn_gate_up(fmt, Wg, Wu, inter, cols, X, act)
    yg, Sg = orc.matvec(fmt, Wg, inter, cols, X)
    yu, Su = orc.matvec(fmt, Wu, inter, cols, X)
    assert np.array_equal(out["g"], yg) and np.array_equal(out["u"], yu)
    assert np.array_equal(out["Sg"], Sg) and np.array_equal(out["Su"], Su)
    f = (lambda t: torch.nn.functional.gelu(t, approximate="tanh")) if act == 1 else torch.nn.functional.silu
    ref = f(torch.tensor(yg)).numpy() * yu
    assert np.allclose(out["h"], ref, rtol=1e-14, atol=0)


def test_ffn_zero_x_and_one_hot(orc):
    fmt, inter, cols = Q4_K, 6, 512
    g_ = synth.rng(13)
    Wg, Wu = synth.q4k(g_, inter, cols), synth.q4k(g_, inter, cols)
    out = orc.ffn_gate_up(fmt, Wg, Wu, inter, cols, np.zeros((1, cols), np.float32), 1)
    assert np.all(out["h"] == 0.0)
    j = 300
    x = np.zeros((1, cols), np.float32)
    x[0, j] = 1.0
    out = orc.ffn_gate_up(fmt, Wg, Wu, inter, cols, x, 2)
    Dg = orc.dequant(fmt, Wg, inter, cols)[:, j].astype(np.float64)
    Du = orc.dequant(fmt, Wu, inter, cols)[:, j].astype(np.float64)
    assert np.allclose(out["h"][0], Dg / (1 + np.exp(-Dg)) * Du, rtol=1e-14, atol=0)


# ---------------------------------------------------------------- MoE routing

def _route_logits(orc, logits, topk):
    """route one token whose logits are given: x = e_0, R[:, 0] = logits."""
    logits = np.asarray(logits, dtype=np.float32)
    E = logits.size
    hidden = 32
    R = np.zeros((E, hidden), np.float32)
    R[:, 0] = logits
    X = np.zeros((1, hidden), np.float32)
    X[0, 0] = 1.0
    return orc.moe_route(R, X, topk)


def test_route_golden_cases(orc):
    for line in golden_lines("moe_rule.txt"):
        lhs, rhs = line.split("->")
        logits = [float(v) for v in lhs.split()]
        expect = [int(v) for v in rhs.split()]
        idx, w, _, _ = _route_logits(orc, logits, len(expect))
        assert idx[0].tolist() == expect


def test_route_renormalised_by_sum_closed_form(orc):
    """top-2 weights are p_a/(p_a+p_b) = 1/(1+exp(l_b-l_a)), not a softmax of p."""
    r = np.random.default_rng(14)
    for _ in range(50):
        l = r.normal(0, 2, 8).astype(np.float32)
        idx, w, lg, _ = _route_logits(orc, l, 2)
        a, b = idx[0]
        la, lb = float(l[a]), float(l[b])
        assert la >= lb
        assert abs(w[0, 0] - 1 / (1 + math.exp(lb - la))) < 1e-14
        assert abs(w[0].sum() - 1) < 1e-15


def test_route_top1_weight_is_one(orc):
    idx, w, _, _ = _route_logits(orc, [0, 0, 0, 0, 0, 100, 0, 0], 1)
    assert idx[0, 0] == 5 and w[0, 0] == 1.0


def test_route_matches_stable_sort(orc):
    """selection = the first k of a stable descending sort (numpy's mergesort),
    including exact ties from repeated small integers."""
    r = np.random.default_rng(15)
    for _ in range(200):
        E = int(r.integers(2, 17))
        k = int(r.integers(1, E + 1))
        l = r.integers(-2, 3, E).astype(np.float32)
        idx, w, _, _ = _route_logits(orc, l, k)
        ref = np.argsort(-l.astype(np.float64), kind="stable")[:k]
        assert idx[0].tolist() == ref.tolist()


def test_route_logits_are_router_dot_x(orc):
    g_ = synth.rng(16)
    R = synth.router(g_, 8, 256)
    X = synth.activations(g_, 5, 256)
    idx, w, lg, labs = orc.moe_route(R, X, 2)
    assert np.allclose(lg, X.astype(np.float64) @ R.T.astype(np.float64), rtol=1e-13, atol=1e-16)
    assert np.allclose(labs, np.abs(X.astype(np.float64)) @ np.abs(R.T.astype(np.float64)), rtol=1e-13)


def _tiny_moe(orc, E=4, hidden=256, inter=512, ntok=3, seed=17):
    g_ = synth.rng(seed)
    W1 = [synth.q4k(g_, inter, hidden) for _ in range(E)]
    W3 = [synth.q4k(g_, inter, hidden) for _ in range(E)]
    W2 = [synth.q4k(g_, hidden, inter) for _ in range(E)]
    X = synth.activations(g_, ntok, hidden)
    return W1, W3, W2, X


def _dense_swiglu(orc, W1, W3, W2, hidden, inter, X):
    f = orc.ffn_gate_up(Q4_K, W1, W3, inter, hidden, X, 2)
    h = f["h"]
    D2 = orc.dequant(Q4_K, W2, hidden, inter).astype(np.float64)
    return h @ D2.T


def test_moe_one_hot_router_equals_single_expert(orc):
    E, hidden, inter = 4, 256, 512
    W1, W3, W2, X = _tiny_moe(orc, E, hidden, inter)
    R = np.zeros((E, hidden), np.float32)
    R[2, :] = 100.0 * np.sign(X[0])          # token 0 strongly prefers expert 2
    idx, w, _, _ = orc.moe_route(R, X[:1], 1)
    assert idx[0, 0] == 2 and w[0, 0] == 1.0
    out = orc.moe_ffn(Q4_K, W1, W3, W2, hidden, inter, X[:1], idx, w)
    ref = _dense_swiglu(orc, W1[2], W3[2], W2[2], hidden, inter, X[:1])
    assert np.allclose(out["Y"], ref, rtol=1e-13, atol=1e-13)


def test_moe_uniform_router_equals_expert_average(orc):
    E, hidden, inter = 4, 256, 512
    W1, W3, W2, X = _tiny_moe(orc, E, hidden, inter, ntok=2)
    R = np.zeros((E, hidden), np.float32)
    idx, w, _, _ = orc.moe_route(R, X, 2)
    assert (idx == [[0, 1], [0, 1]]).all() and (w == 0.5).all()
    out = orc.moe_ffn(Q4_K, W1, W3, W2, hidden, inter, X, idx, w)
    y0 = _dense_swiglu(orc, W1[0], W3[0], W2[0], hidden, inter, X)
    y1 = _dense_swiglu(orc, W1[1], W3[1], W2[1], hidden, inter, X)
    assert np.allclose(out["Y"], 0.5 * (y0 + y1), rtol=1e-13, atol=1e-13)


def test_moe_scalar_reference(orc):
    """random routing: Y_t = sum_k w_tk * (dense SwiGLU FFN of expert idx[t,k])(x_t)."""
    E, hidden, inter, ntok = 4, 256, 512, 3
    W1, W3, W2, X = _tiny_moe(orc, E, hidden, inter, ntok, seed=18)
    R = synth.router(synth.rng(19), E, hidden) * 50
    idx, w, _, _ = orc.moe_route(R, X, 2)
    out = orc.moe_ffn(Q4_K, W1, W3, W2, hidden, inter, X, idx, w)
    for t in range(ntok):
        ref = sum(w[t, k] * _dense_swiglu(orc, W1[idx[t, k]], W3[idx[t, k]], W2[idx[t, k]],
                                          hidden, inter, X[t:t + 1])[0] for k in range(2))
        assert np.allclose(out["Y"][t], ref, rtol=1e-13, atol=1e-13)
        for k in range(2):
            ye = _dense_swiglu(orc, W1[idx[t, k]], W3[idx[t, k]], W2[idx[t, k]], hidden, inter,
                               X[t:t + 1])[0]
            assert np.allclose(out["ye"][t * 2 + k], ye, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- input RMS-norm

def test_rmsnorm_pins(orc):
    """x * w / sqrt(mean(x^2) + eps) against torch's rms_norm, a constant
    row's closed form, scale invariance at eps = 0, unit mean square at unit
    weight, and linearity in the weight."""
    n = 2560
    X = synth.activations(synth.rng(60), 3, n) * np.float32(3.0)
    w = (1.0 + 0.1 * synth.activations(synth.rng(61), 1, n)[0]).astype(np.float32)
    for eps in (1e-6, 1e-5):
        got = orc.rmsnorm(X, w, eps)
        ref = torch.nn.functional.rms_norm(torch.tensor(X, dtype=torch.float64), (n,),
                                           torch.tensor(w, dtype=torch.float64), eps).numpy()
        assert np.allclose(got, ref, rtol=1e-14, atol=1e-15)
    c = np.full((1, n), -2.5, np.float32)
    ones = np.ones(n, np.float32)
    assert np.allclose(orc.rmsnorm(c, ones, 1e-5), -2.5 / math.sqrt(6.25 + 1e-5), rtol=1e-15, atol=0)
    u = orc.rmsnorm(X, ones, 0.0)
    assert np.allclose((u ** 2).mean(axis=1), 1.0, rtol=1e-14)
    assert np.allclose(orc.rmsnorm(X * np.float32(8.0), ones, 0.0), u, rtol=1e-14, atol=0)   # 8x is exact in fp32
    assert np.allclose(orc.rmsnorm(X, w * np.float32(2.0), 1e-6), 2 * orc.rmsnorm(X, w, 1e-6), rtol=1e-15, atol=0)


# ---------------------------------------------------------------- MoE variants
# dotLLM PR #320 Qwen-MoE commit (norm_topk_prob = false, shared expert with
# an optional sigmoid gate) and its N-shared-experts follow-up.

def test_moe_weights_raw(orc):
    """norm_topk_prob = false: the selected softmax probabilities themselves."""
    rng = np.random.default_rng(40)
    lg = rng.normal(0, 2, (6, 8))
    idx = np.argsort(-lg, axis=1, kind="stable")[:, :2].astype(np.int32)
    raw = orc.moe_weights(lg, idx, norm=False)
    p = torch.softmax(torch.tensor(lg), dim=-1).numpy()
    assert np.allclose(raw, np.take_along_axis(p, idx, 1), rtol=1e-14, atol=0)
    # renormalising the raw weights gives the (pinned) renormalised rule
    assert np.allclose(orc.moe_weights(lg, idx), raw / raw.sum(1, keepdims=True), rtol=1e-14, atol=0)
    # uniform logits: 1/E each; two experts, top-1: the logistic of the logit gap
    assert np.allclose(orc.moe_weights(np.zeros((1, 8)), np.array([[3, 5]], np.int32), norm=False), 1 / 8,
                       rtol=1e-15, atol=0)
    from scipy.special import expit
    two = np.array([[1.7, -0.4]])
    assert abs(orc.moe_weights(two, np.array([[0]], np.int32), norm=False)[0, 0] - expit(2.1)) < 1e-15


def _shared_mats(seed, hidden=256, inter=512):
    g_ = synth.rng(seed)
    return synth.q4k(g_, inter, hidden), synth.q4k(g_, inter, hidden), synth.q4k(g_, hidden, inter)


def test_moe_shared_single_expert_is_dense_swiglu(orc):
    hidden, inter = 256, 512
    Wg, Wu, Wd = _shared_mats(41)
    X = synth.activations(synth.rng(42), 3, hidden)
    S, gs = orc.moe_shared(Q4_K, [Wg], [Wu], [Wd], hidden, inter, X)
    assert (gs == 1.0).all()
    assert np.allclose(S, _dense_swiglu(orc, Wg, Wu, Wd, hidden, inter, X), rtol=1e-13, atol=1e-13)


def test_moe_shared_experts_sum(orc):
    """N shared experts are summed: two distinct ones give the sum of each,
    two identical ones twice one (the follow-up commit's unit tests)."""
    hidden, inter = 256, 512
    a, b = _shared_mats(43), _shared_mats(44)
    X = synth.activations(synth.rng(45), 2, hidden)
    one = lambda m: orc.moe_shared(Q4_K, [m[0]], [m[1]], [m[2]], hidden, inter, X)[0]
    both, _ = orc.moe_shared(Q4_K, [a[0], b[0]], [a[1], b[1]], [a[2], b[2]], hidden, inter, X)
    assert np.allclose(both, one(a) + one(b), rtol=1e-13, atol=1e-13)
    twice, _ = orc.moe_shared(Q4_K, [a[0], a[0]], [a[1], a[1]], [a[2], a[2]], hidden, inter, X)
    assert np.array_equal(twice, 2 * one(a))


def test_moe_shared_gate(orc):
    """sigmoid(g . x) scales the branch: g = 0 halves it exactly, large
    |g . x| saturates to 0 or 1, and random g agrees with the library logistic."""
    from scipy.special import expit
    hidden, inter = 256, 512
    Wg, Wu, Wd = _shared_mats(46)
    X = synth.activations(synth.rng(47), 2, hidden)
    ungated, _ = orc.moe_shared(Q4_K, [Wg], [Wu], [Wd], hidden, inter, X)
    half, gs = orc.moe_shared(Q4_K, [Wg], [Wu], [Wd], hidden, inter, X, gate=np.zeros(hidden, np.float32))
    assert (gs == 0.5).all() and np.array_equal(half, 0.5 * ungated)
    big = (50.0 * np.sign(X[0])).astype(np.float32)
    hi, gs = orc.moe_shared(Q4_K, [Wg], [Wu], [Wd], hidden, inter, X[:1], gate=big)
    lo, gs2 = orc.moe_shared(Q4_K, [Wg], [Wu], [Wd], hidden, inter, X[:1], gate=-big)
    assert gs[0] == 1.0 and np.array_equal(hi, ungated[:1]) and gs2[0] < 1e-300 and np.abs(lo).max() < 1e-290
    g = synth.activations(synth.rng(48), 1, hidden)[0] * np.float32(0.05)
    _, gs = orc.moe_shared(Q4_K, [Wg], [Wu], [Wd], hidden, inter, X, gate=g)
    assert np.allclose(gs, expit(X.astype(np.float64) @ g.astype(np.float64)), rtol=1e-14, atol=0)


def test_moe_shared_zero_down_adds_nothing(orc):
    hidden, inter = 256, 512
    Wg, Wu, _ = _shared_mats(49)
    Wd0 = np.zeros((hidden, inter // 256 * 144), np.uint8)     # d = dmin = 0: every weight 0
    X = synth.activations(synth.rng(50), 2, hidden)
    S, _ = orc.moe_shared(Q4_K, [Wg], [Wu], [Wd0], hidden, inter, X)
    assert (S == 0).all()


def test_abs_matvec(orc):
    W, _ = _mat(Q6_K, 5, 512, seed=20)
    D = np.abs(orc.dequant(Q6_K, W, 5, 512).astype(np.float64))
    v = np.random.default_rng(21).uniform(0, 1, 512)
    assert np.allclose(orc.abs_matvec(Q6_K, W, 5, 512, v), D @ v, rtol=1e-13)


def test_moe_weights_of_selection(orc):
    """weights of a given selection: equal to the router's own when the selection
    is the router's; renormalised by the selected sum for any other selection."""
    g_ = synth.rng(22)
    R = synth.router(g_, 8, 256) * 20
    X = synth.activations(g_, 6, 256)
    idx, w, lg, _ = orc.moe_route(R, X, 2)
    assert np.allclose(orc.moe_weights(lg, idx), w, rtol=1e-15, atol=0)
    other = np.array([[3, 1]] * 6, dtype=np.int32)
    wo = orc.moe_weights(lg, other)
    for t in range(6):
        assert abs(wo[t, 0] - 1 / (1 + math.exp(lg[t, 1] - lg[t, 3]))) < 1e-14


def test_dense_matvec_pins():
    """dense_matvec against closed forms: the identity returns x, an all-ones
    fp16 matrix returns each row's sum of x, a one-hot row picks one column,
    and fp16 values go in exactly (2^-24 survives where an fp16-rounded x
    product would not)."""
    import oracle
    g = np.random.default_rng(5)
    x = g.standard_normal((2, 64)).astype(np.float32)
    y, S = oracle.dense_matvec(np.eye(64, dtype=np.float32), x)
    assert np.array_equal(y, x.astype(np.float64)) and np.array_equal(S, np.abs(x.astype(np.float64)))
    y, _ = oracle.dense_matvec(np.ones((3, 64), np.float16), x)
    assert np.allclose(y, np.repeat(x.astype(np.float64).sum(axis=1, keepdims=True), 3, axis=1), rtol=0, atol=1e-12)
    W = np.zeros((5, 64), np.float16)
    W[2, 17] = np.float16(-2.5)
    y, _ = oracle.dense_matvec(W, x)
    assert y[0, 2] == -2.5 * float(x[0, 17]) and (np.delete(y[0], 2) == 0).all()
    W = np.full((1, 4), np.float16(2.0 ** -24))          # the smallest fp16 subnormal
    y, _ = oracle.dense_matvec(W, np.ones((1, 4), np.float32))
    assert y[0, 0] == 4 * 2.0 ** -24

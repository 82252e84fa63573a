"""GPU parity at the full sizes of the named workloads, through the same C-ABI
calls the benchmark times (batch 1 decode layer; Llama FFN at batch 1..8;
lm_head; Mixtral MoE).  Outputs the oracle can afford are checked in full;
the larger ones on seeded row samples (first and last rows included)."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

Q4_K, Q6_K, Q8_0 = 1, 2, 3
GEGLU, SWIGLU = 1, 2
NTH = oracle.threads_default()


@pytest.fixture(scope="module")
def lq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_weight_super_gb300 as pkg
    from block_quantized_weight_super_gb300 import build
    build.build()
    pkg.lib()
    yield pkg
    from gpu_util import status_clean
    status_clean(pkg)


from gpu_util import assert_within, dev, empty, host  # noqa: E402


def _sample_rows(n, k, seed):
    g = np.random.default_rng(seed)
    idx = np.unique(np.concatenate([[0, n - 1], g.choice(n, size=min(k, n), replace=False)]))
    return idx.astype(np.int64)


def _act(a, act):
    f = oracle.gelu_tanh if act == GEGLU else oracle.silu
    return np.vectorize(f, otypes=[np.float64])(a)


def _check_gate_up_rows(fmt, Wg, Wu, cols, x, h_gpu, rows, act):
    g, Sg = oracle.matvec_rows(fmt, Wg, cols, rows, x, NTH)
    u, Su = oracle.matvec_rows(fmt, Wu, cols, rows, x, NTH)
    ref = _act(g, act) * u
    assert_within(h_gpu[:, rows], ref, oracle.gate_up_bound(g, u, Sg, Su, act), "gate_up rows")


def test_matvec_small_workload(lq):
    """single Q4_K matvec 256 x 2560, batch 1 (all outputs)."""
    W, x = synth.matvec_small(0)
    y = empty((1, 256))
    lq.lq_matvec(Q4_K, dev(W), 256, 2560, dev(x), y, 1)
    ref, S = oracle.matvec(Q4_K, W, 256, 2560, x, NTH)
    assert_within(host(y), ref, oracle.matvec_bound(S), "matvec_small")


def test_gemma3_decode_layer(lq):
    """the benchmark's layer at full size: mixed QKV, O, fused gate+up GEGLU,
    Q6_K down (each fed the GPU's own input, so the per-call bound applies)."""
    L, x = synth.gemma3_layer(0)
    H, I, NQ, NKV = synth.GEMMA3_HIDDEN, synth.GEMMA3_INTER, synth.GEMMA3_NQ, synth.GEMMA3_NKV
    d = {k: dev(v) for k, v in L.items()}
    xd = dev(x)
    q, k, v = empty((1, NQ)), empty((1, NKV)), empty((1, NKV))
    lq.lq_qkv_mixed(Q4_K, d["wq"], NQ, Q4_K, d["wk"], NKV, Q6_K, d["wv"], NKV, H, xd, q, k, v, 1)
    for name, fmt, W, n, out in (("q", Q4_K, L["wq"], NQ, q), ("k", Q4_K, L["wk"], NKV, k),
                                 ("v", Q6_K, L["wv"], NKV, v)):
        ref, S = oracle.matvec(fmt, W, n, H, x, NTH)
        assert_within(host(out), ref, oracle.matvec_bound(S), "qkv " + name)
    o = empty((1, H))
    lq.lq_matvec(Q4_K, d["wo"], H, NQ, q, o, 1)
    qh = host(q)
    ref, S = oracle.matvec(Q4_K, L["wo"], H, NQ, qh, NTH)
    assert_within(host(o), ref, oracle.matvec_bound(S), "o")
    rb = lq.lq_row_bytes(Q4_K, H)
    wgu = torch.empty(2 * I * rb, dtype=torch.uint8, device="cuda")
    lq.lq_pack_gate_up(Q4_K, d["wg"], d["wu"], I, H, wgu)
    h = empty((1, I))
    lq.lq_ffn_gate_up_act(Q4_K, wgu, I, H, o, h, 1, GEGLU)
    oh = host(o)
    r = oracle.ffn_gate_up(Q4_K, L["wg"], L["wu"], I, H, oh, GEGLU, NTH)
    hh = host(h)
    assert_within(hh, r["h"], oracle.gate_up_bound(r["g"], r["u"], r["Sg"], r["Su"], GEGLU), "gate_up")
    y = empty((1, H))
    lq.lq_matvec(Q6_K, d["wd"], H, I, h, y, 1)
    ref, S = oracle.matvec(Q6_K, L["wd"], H, I, hh, NTH)
    assert_within(host(y), ref, oracle.matvec_bound(S), "down")


@pytest.mark.parametrize("fmt", [Q4_K, Q8_0])
@pytest.mark.parametrize("batch", [1, 2, 4, 8])
def test_llama_ffn_workload(lq, fmt, batch):
    """SwiGLU FFN 2 x 14336 x 4096 + down 4096 x 14336 at batch 1..8, sampled rows."""
    W, X = synth.llama_ffn(fmt, batch, seed=batch)
    H, I = synth.LLAMA_HIDDEN, synth.LLAMA_INTER
    rb = lq.lq_row_bytes(fmt, H)
    wgu = torch.empty(2 * I * rb, dtype=torch.uint8, device="cuda")
    lq.lq_pack_gate_up(fmt, dev(W["wg"]), dev(W["wu"]), I, H, wgu)
    h = empty((batch, I))
    lq.lq_ffn_gate_up_act(fmt, wgu, I, H, dev(X), h, batch, SWIGLU)
    hh = host(h)
    assert np.isfinite(hh).all()
    _check_gate_up_rows(fmt, W["wg"], W["wu"], H, X, hh, _sample_rows(I, 384, 11 + batch), SWIGLU)
    y = empty((batch, H))
    lq.lq_matvec(fmt, dev(W["wd"]), H, I, h, y, batch)
    rows = _sample_rows(H, 384, 23 + batch)
    ref, S = oracle.matvec_rows(fmt, W["wd"], I, rows, hh, NTH)
    assert_within(host(y)[:, rows], ref, oracle.matvec_bound(S), "down rows")


def test_lm_head_workload(lq):
    """262144 x 2560 Q4_K logits of an RMS-normed x, batch 1, sampled rows."""
    W, x = synth.lm_head(0)
    V, H = W.shape[0], synth.GEMMA3_HIDDEN
    y = empty((1, V))
    lq.lq_matvec(Q4_K, dev(W), V, H, dev(x), y, 1)
    yh = host(y)
    assert np.isfinite(yh).all()
    rows = _sample_rows(V, 2048, 5)
    ref, S = oracle.matvec_rows(Q4_K, W, H, rows, x, NTH)
    assert_within(yh[:, rows], ref, oracle.matvec_bound(S), "lm_head rows")


def test_mixtral_moe_workload(lq):
    """8 experts of 14336 x 4096 Q4_K, top-2, 16 tokens (all outputs)."""
    R, W1, W3, W2, X = synth.mixtral_moe(0)
    E, hidden = R.shape
    inter, ntok, topk = W1[0].shape[0], X.shape[0], synth.MIXTRAL_TOPK
    Y = empty((ntok, hidden))
    idx = torch.full((ntok, topk), -1, dtype=torch.int32, device="cuda")
    w = empty((ntok, topk))
    nbytes = lq.lq_moe_workspace_bytes(E, topk, ntok, hidden, inter)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d1, d3, d2 = [dev(a) for a in W1], [dev(a) for a in W3], [dev(a) for a in W2]
    lq.lq_moe_ffn(dev(R), E, topk, Q4_K, d1, d3, d2, hidden, inter, dev(X), Y, ntok, idx, w, ws, nbytes)
    idx_h = host(idx)
    _, _, lg, labs = oracle.moe_route(R, X, topk)
    chk = oracle.moe_check(Q4_K, W1, W3, W2, hidden, inter, X, lg, labs, idx_h, NTH)
    assert chk["admissible"].all()
    elmax = chk["el"].max(axis=1, keepdims=True)
    assert_within(host(w), chk["w"], 2 * chk["w"] * elmax + 8 * oracle.U32, "moe weights")
    assert_within(host(Y), chk["Y"], chk["bound"], "moe Y")

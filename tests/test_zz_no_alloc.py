"""lq_moe_ffn_static (static device scratch, no allocation) against
lq_moe_ffn with a caller workspace, over two calls in a row on different
inputs, within the MoE parity bound of the oracle.  Collected last (file
name) so it also runs after every other test in one process."""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

Q4_K = 1
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


def _case(seed, E, topk, ntok, hidden, inter):
    R, W1, W3, W2, X = synth.mixtral_moe(seed, E, hidden, inter, ntok)
    return R, W1, W3, W2, X


def _call(lq, fn, R, W1, W3, W2, X, topk, E, hidden, inter, ntok):
    Y = empty((ntok, hidden))
    idx = torch.full((ntok, topk), -1, dtype=torch.int32, device="cuda")
    w = empty((ntok, topk))
    d1, d3, d2 = [dev(a) for a in W1], [dev(a) for a in W3], [dev(a) for a in W2]
    if fn == "static":
        lq.lq_moe_ffn_static(dev(R), E, topk, Q4_K, d1, d3, d2, hidden, inter, dev(X), Y, ntok, idx, w)
    else:
        nbytes = lq.lq_moe_workspace_bytes(E, topk, ntok, hidden, inter)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        lq.lq_moe_ffn(dev(R), E, topk, Q4_K, d1, d3, d2, hidden, inter, dev(X), Y, ntok, idx, w, ws, nbytes)
    torch.cuda.synchronize()
    return host(Y), host(idx), host(w)


def test_static_scratch_matches_workspace_entry_point_twice(lq):
    E, topk, hidden, inter = 8, 2, 256, 512
    cases = [_case(71, E, topk, 6, hidden, inter), _case(72, E, topk, 11, hidden, inter)]
    for R, W1, W3, W2, X in cases:                  # two calls in a row, different shapes
        ntok = X.shape[0]
        Ys, idx_s, w_s = _call(lq, "static", R, W1, W3, W2, X, topk, E, hidden, inter, ntok)
        Yw, idx_w, w_w = _call(lq, "workspace", R, W1, W3, W2, X, topk, E, hidden, inter, ntok)
        _, _, lg, labs = oracle.moe_route(R, X, topk)
        chk = oracle.moe_check(Q4_K, W1, W3, W2, hidden, inter, X, lg, labs, idx_w, NTH)
        assert np.array_equal(idx_s, idx_w)
        elmax = chk["el"].max(axis=1, keepdims=True)
        assert_within(w_s, w_w, 2 * chk["w"] * elmax + 8 * oracle.U32, "static vs workspace weights")
        assert_within(Ys, Yw, chk["bound"], "static vs workspace Y")
        assert_within(Ys, chk["Y"], chk["bound"], "static vs oracle Y")


def test_static_scratch_rejects_oversized_shapes(lq):
    E, topk, hidden, inter = 4, 2, 4096, 14336
    ntok = 64                                        # 64 * 2 rows * (4096 + 14336) * 4 B > 4 MiB
    need = lq.lq_moe_workspace_bytes(E, topk, ntok, hidden, inter)
    assert need > lq.LQ_MOE_STATIC_SCRATCH_BYTES
    W = [torch.zeros(inter * hidden // 256 * 144, dtype=torch.uint8, device="cuda")] * E
    W2 = [torch.zeros(hidden * inter // 256 * 144, dtype=torch.uint8, device="cuda")] * E
    R = torch.zeros((E, hidden), device="cuda")
    X = torch.zeros((ntok, hidden), device="cuda")
    Y = torch.zeros((ntok, hidden), device="cuda")
    with pytest.raises(lq.LqError) as ei:
        lq.lq_moe_ffn_static(R, E, topk, Q4_K, W, W, W2, hidden, inter, X, Y, ntok)
    assert ei.value.status == lq.LQ_EWORKSPACE
    assert "static scratch" in lq.lq_last_error()


def _static_args(lq, case, topk, E, hidden, inter):
    R, W1, W3, W2, X = case
    ntok = X.shape[0]
    d = {"R": dev(R), "W1": [dev(a) for a in W1], "W3": [dev(a) for a in W3], "W2": [dev(a) for a in W2],
         "X": dev(X), "Y": empty((ntok, hidden)), "idx": torch.full((ntok, topk), -1, dtype=torch.int32, device="cuda"),
         "w": empty((ntok, topk)), "ntok": ntok}
    return d


def _static(lq, d, topk, E, hidden, inter, stream=None):
    lq.lq_moe_ffn_static(d["R"], E, topk, Q4_K, d["W1"], d["W3"], d["W2"], hidden, inter, d["X"], d["Y"],
                         d["ntok"], d["idx"], d["w"], stream=stream)


def _workspace(lq, d, topk, E, hidden, inter):
    nbytes = lq.lq_moe_workspace_bytes(E, topk, d["ntok"], hidden, inter)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    Y = empty((d["ntok"], hidden))
    lq.lq_moe_ffn(d["R"], E, topk, Q4_K, d["W1"], d["W3"], d["W2"], hidden, inter, d["X"], Y, d["ntok"], None, None,
                  ws, nbytes)
    return host(Y)


def test_static_back_to_back_shapes_one_stream(lq):
    """Two static calls of different shapes queued on one stream with no
    synchronisation between them (the scratch is reused in stream order),
    each equal to the workspace entry point's result bit for bit (same
    kernels, same scratch layout)."""
    E, topk, hidden, inter = 8, 2, 256, 512
    a = _static_args(lq, _case(81, E, topk, 6, hidden, inter), topk, E, hidden, inter)
    b = _static_args(lq, _case(82, E, topk, 13, hidden, inter), topk, E, hidden, inter)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        _static(lq, a, topk, E, hidden, inter, st)
        _static(lq, b, topk, E, hidden, inter, st)
    st.synchronize()
    for d in (a, b):
        assert np.array_equal(host(d["Y"]), _workspace(lq, d, topk, E, hidden, inter))


def test_static_near_the_scratch_limit(lq):
    """hidden 4096, inter 14336 at 56 routed rows (two experts, top-2, 28
    tokens): 4,130,304 of the 4,194,304 scratch bytes.  Equal to the
    workspace entry point bit for bit; three tokens checked against the
    oracle."""
    E, topk, ntok, hidden, inter = 2, 2, 28, 4096, 14336
    need = lq.lq_moe_workspace_bytes(E, topk, ntok, hidden, inter)
    assert lq.LQ_MOE_STATIC_SCRATCH_BYTES - 65536 < need <= lq.LQ_MOE_STATIC_SCRATCH_BYTES
    case = _case(83, E, topk, ntok, hidden, inter)
    d = _static_args(lq, case, topk, E, hidden, inter)
    _static(lq, d, topk, E, hidden, inter)
    Ys = host(d["Y"])
    assert np.array_equal(Ys, _workspace(lq, d, topk, E, hidden, inter))
    R, W1, W3, W2, X = case
    for t in (0, 13, ntok - 1):
        _, _, lg, labs = oracle.moe_route(R, X[t:t + 1], topk)
        chk = oracle.moe_check(Q4_K, W1, W3, W2, hidden, inter, X[t:t + 1], lg, labs, host(d["idx"])[t:t + 1], NTH)
        assert_within(Ys[t:t + 1], chk["Y"], chk["bound"], f"near-limit token {t}")


def test_static_call_captures_in_a_graph_without_allocating(lq):
    """After a first (set-up) call, a static call captures into a CUDA graph
    under the global capture mode (any allocation during capture would fail
    the capture) and an eager static call leaves the device's free memory
    unchanged; the graph's replay equals the eager result bit for bit."""
    E, topk, hidden, inter = 4, 2, 256, 512
    d = _static_args(lq, _case(84, E, topk, 9, hidden, inter), topk, E, hidden, inter)
    _static(lq, d, topk, E, hidden, inter)          # set-up call
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    _static(lq, d, topk, E, hidden, inter)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    ref = host(d["Y"]).copy()
    d["Y"].fill_(float("nan"))
    st = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st, capture_error_mode="global"):
        _static(lq, d, topk, E, hidden, inter, st)
    torch.cuda.synchronize()
    assert np.isnan(host(d["Y"])).all()              # capture ran nothing
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host(d["Y"]), ref)

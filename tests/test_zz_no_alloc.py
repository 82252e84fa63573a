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

"""Tail-skip on the decode kernels (PolyStrata, "Models and backends",
section "What was tuned") against the oracle's tail-skip: an expert every
token of a call ranks at place n + 1 or later of its picks is not computed,
the other picks keep their weights, and a prompt batch is not touched.
Floats within the parity bars (rel-L2 5e-3, max-abs 2e-2 * rms of the
reference beyond the bf16 output's own rounding); the published weights of
left-out picks are exactly 0."""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_fwd_gb300 as q
from tests import gpu_util as G
from workloads import gen

pytestmark = pytest.mark.gpu

DIMS = gen.QWEN
_L = {}


def layer():
    if "l" not in _L:
        planes = gen.draw_layer(DIMS, 21)
        _L["l"] = (planes, q.DeviceLayer(planes, G.dev()))
    return _L["l"]


def tokens(T, seed):
    return oracle.rmsnorm(gen.draw_tokens(DIMS, T, seed, "resid"))


def run(dl, xb, n, forced=None):
    T = xb.shape[0]
    out = torch.full((T, DIMS.hidden), -1, dtype=torch.int16, device=G.dev())
    ids = torch.empty((T, DIMS.top_k), dtype=torch.int32, device=G.dev())
    w = torch.empty((T, DIMS.top_k), dtype=torch.float32, device=G.dev())
    ws = q.make_workspace(DIMS, T, G.dev())
    fi, fw = (None, None) if forced is None else (G.i32(forced[0]), G.f32(forced[1]))
    q.moe_layer_forward_tail_skip(DIMS, dl, G.u16(xb), out, ws, n, forced_ids=fi,
                                  forced_weights=fw, ids=ids, weights=w)
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    return G.bf16_to_np(out), ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T", [1, 2, 4, 16, 32])
@pytest.mark.parametrize("n", [5, 7])
def test_forced_routing(T, n):
    planes, dl = layer()
    xb = tokens(T, 100 + T)
    ref = oracle.moe_forward(DIMS, planes, xb)
    w2, sk = oracle.tail_skip(ref["ids"], ref["w"], n)
    assert sk.any()
    want = oracle.moe_forward(DIMS, planes, xb, ids=ref["ids"], w=w2)
    out, ids, w = run(dl, xb, n, forced=(ref["ids"], ref["w"]))
    assert np.array_equal(ids, ref["ids"])
    assert np.array_equal(w, w2)                      # kept as given, left out exactly 0
    G.assert_close(out, want["out"], f"tail-skip {n} T={T}, forced")


def test_own_routing_single_token():
    """T = 1, n = 7: the token's lowest-weight pick is left out.  Tokens whose
    two lowest weights are within 1e-3 of each other would make the choice a
    near tie and are drawn past."""
    planes, dl = layer()
    seed = 0
    for seed in range(40):
        xb = tokens(1, 300 + seed)
        ref = oracle.moe_forward(DIMS, planes, xb)
        ws_ = np.sort(ref["w"][0])
        if ref["gap"][0] >= 1e-4 and ws_[1] - ws_[0] > 1e-3 * ws_[1]:
            break
    w2, sk = oracle.tail_skip(ref["ids"], ref["w"], 7)
    want = oracle.moe_forward(DIMS, planes, xb, ids=ref["ids"], w=w2)
    out, ids, w = run(dl, xb, 7)
    assert np.array_equal(ids, ref["ids"])
    assert np.array_equal(w == 0.0, sk)
    np.testing.assert_allclose(w[~sk], ref["w"][~sk], rtol=1e-4, atol=1e-6)
    G.assert_close(out, want["out"], "tail-skip 7 T=1, own routing")


@pytest.mark.parametrize("n", [0, 8, 9])
def test_off_is_the_plain_layer(n):
    planes, dl = layer()
    xb = tokens(4, 7)
    ref = oracle.moe_forward(DIMS, planes, xb)
    out, ids, w = run(dl, xb, n, forced=(ref["ids"], ref["w"]))
    assert np.array_equal(w, ref["w"])
    G.assert_close(out, ref["out"], f"tail-skip {n} (off)")
    # at T = 1 the plain layer runs the same decode kernels: bit for bit
    x1 = tokens(1, 8)
    out1, _, _ = run(dl, x1, n)
    plain = torch.empty((1, DIMS.hidden), dtype=torch.int16, device=G.dev())
    q.moe_layer_forward(DIMS, dl, G.u16(x1), plain, q.make_workspace(DIMS, 1, G.dev()))
    torch.cuda.synchronize()
    assert np.array_equal(out1, G.bf16_to_np(plain))


def test_prompt_batch_is_not_touched():
    planes, dl = layer()
    T = 64
    xb = tokens(T, 9)
    out, _, w = run(dl, xb, 5)
    plain = torch.empty((T, DIMS.hidden), dtype=torch.int16, device=G.dev())
    q.moe_layer_forward(DIMS, dl, G.u16(xb), plain, q.make_workspace(DIMS, T, G.dev()))
    torch.cuda.synchronize()
    assert np.array_equal(out, G.bf16_to_np(plain))
    assert (w > 0).all()

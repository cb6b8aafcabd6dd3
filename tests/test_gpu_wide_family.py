"""Parity of the whole layer on the wider expert geometry of the model family
the pages also serve (Flash-Next: 512 routed experts a layer; the write-ups
give the expert count, not the rest of the shape, so the Qwen3.6 hidden and
intermediate sizes are kept and top-10 is taken as the pick count).  Each
token count is on a different path: T = 1, 2 on the decode kernels, T = 4
and T = 300 on the tcgen05 kernels, plus the decode kernels' stage calls at
T = 12.  Same bars as the other parity tests: ids bit-exact away from near
ties, floats within rel-L2 5e-3 and max-abs 2e-2 * rms(ref)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_fwd_gb300 as q
from tests import gpu_util as G
from workloads import gen

pytestmark = pytest.mark.gpu

WIDE = gen.LayerDims(hidden=2048, n_experts=512, top_k=10, inter=512, shared_inter=512)

_LAYER = {}


def layer():
    if "l" not in _LAYER:
        planes = gen.draw_layer(WIDE, 3)
        _LAYER["l"] = (planes, q.DeviceLayer(planes, G.dev()))
    return _LAYER["l"]


@pytest.mark.parametrize("T", [1, 2, 4, 300])
def test_wide_family_layer(T):
    planes, dl = layer()
    xb = oracle.rmsnorm(gen.draw_tokens(WIDE, T, 11 + T, "resid"))
    ref = oracle.moe_forward(WIDE, planes, xb)
    x = G.u16(xb)
    out = torch.full((T, WIDE.hidden), -1, dtype=torch.int16, device=G.dev())
    ids = torch.empty((T, WIDE.top_k), dtype=torch.int32, device=G.dev())
    w = torch.empty((T, WIDE.top_k), dtype=torch.float32, device=G.dev())
    sig = torch.empty((T,), dtype=torch.float32, device=G.dev())
    ws = q.make_workspace(WIDE, T, G.dev())
    q.moe_layer_forward(WIDE, dl, x, out, ws, ids=ids, weights=w, shared_gate=sig)
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    clear = G.clear_tokens(ref["gap"])
    assert np.array_equal(ids.cpu().numpy()[clear], ref["ids"][clear])
    assert np.allclose(w.cpu().numpy()[clear], ref["w"][clear], rtol=1e-4, atol=1e-6)
    assert np.allclose(sig.cpu().numpy(), ref["sig"], rtol=1e-4, atol=1e-6)
    G.assert_close(G.bf16_to_np(out)[clear], ref["out"][clear], f"E=512 K=10 T={T}")
    if len(clear) < T:
        out2 = torch.full_like(out, -1)
        q.moe_layer_forward_routed(WIDE, dl, x, G.i32(ref["ids"]), G.f32(ref["w"]), out2, ws)
        torch.cuda.synchronize()
        assert q.moe_get_device_status(ws) == q.STRATA_OK
        G.assert_close(G.bf16_to_np(out2), ref["out"], f"E=512 K=10 T={T}, forced routing")


def test_wide_family_decode_stage_calls():
    """T = 12 (120 pairs) through moe_decode_route -> moe_decode_gate_up ->
    moe_decode_down_combine, the calls that keep the decode kernels up to
    32 tokens: own routing, then the oracle's routing forced."""
    planes, dl = layer()
    T = 12
    xb = oracle.rmsnorm(gen.draw_tokens(WIDE, T, 5, "resid"))
    ref = oracle.moe_forward(WIDE, planes, xb)
    clear = G.clear_tokens(ref["gap"])
    x = G.u16(xb)
    ws = q.make_workspace(WIDE, T, G.dev())
    for forced in (False, True):
        out = torch.full((T, WIDE.hidden), -1, dtype=torch.int16, device=G.dev())
        ids = torch.empty((T, WIDE.top_k), dtype=torch.int32, device=G.dev())
        q.moe_decode_route(WIDE, dl, x, ws, forced=forced)
        if forced:
            q.moe_decode_gate_up(WIDE, dl, x, ws, forced_ids=G.i32(ref["ids"]),
                                 forced_weights=G.f32(ref["w"]), ids=ids)
        else:
            q.moe_decode_gate_up(WIDE, dl, x, ws, ids=ids)
        q.moe_decode_down_combine(WIDE, dl, T, out, ws)
        torch.cuda.synchronize()
        assert q.moe_get_device_status(ws) == q.STRATA_OK
        got = G.bf16_to_np(out)
        if forced:
            assert np.array_equal(ids.cpu().numpy(), ref["ids"])
            G.assert_close(got, ref["out"], "E=512 K=10 T=12 decode kernels, forced")
        else:
            assert np.array_equal(ids.cpu().numpy()[clear], ref["ids"][clear])
            G.assert_close(got[clear], ref["out"][clear], "E=512 K=10 T=12 decode kernels")

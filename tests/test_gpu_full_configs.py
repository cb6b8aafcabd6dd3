"""Parity at the full sizes of the workloads, in the launch configuration the
bench times: the prefill layer at T=2048 (Zipf routing) and the 40-layer
decode stack at T=1 and T=4."""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_fwd_gb300 as q
from tests import gpu_util as G
from workloads import gen

pytestmark = pytest.mark.gpu


def test_prefill_T2048_zipf_full_size():
    cfg = gen.CONFIGS["prefill"]
    dims, T = cfg.dims, cfg.tokens
    planes = gen.draw_layer(dims, 0, bias=cfg.bias, alpha=cfg.alpha)
    dl = q.DeviceLayer(planes, G.dev())
    xb = oracle.rmsnorm(gen.draw_tokens(dims, T, 0, cfg.token_kind))
    ref = oracle.moe_forward(dims, planes, xb)
    x = G.u16(xb)
    out = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
    ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=G.dev())
    ws = q.make_workspace(dims, T, G.dev())
    q.moe_layer_forward(dims, dl, x, out, ws, ids=ids)
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    clear = G.clear_tokens(ref["gap"])
    assert len(clear) >= T - 8
    got_ids = ids.cpu().numpy()
    assert np.array_equal(got_ids[clear], ref["ids"][clear])
    got = G.bf16_to_np(out)
    G.assert_close(got[clear], ref["out"][clear], "prefill T=2048")
    # expert loads span the skew the workload asks for
    loads = np.bincount(ref["ids"].ravel(), minlength=dims.n_experts)
    assert loads.max() >= 250
    if len(clear) < T:
        out2 = torch.empty_like(out)
        q.moe_layer_forward_routed(dims, dl, x, G.i32(ref["ids"]), G.f32(ref["w"]), out2, ws)
        torch.cuda.synchronize()
        G.assert_close(G.bf16_to_np(out2), ref["out"], "prefill T=2048, forced routing")


_STACK = {}


def stack_layers(n):
    """The stack workload's layers (seeds 0..39), and more with the next
    seeds, drawn once per test session."""
    dims = gen.QWEN
    seeds = list(gen.CONFIGS["stack"].seeds)
    seeds += list(range(seeds[-1] + 1, seeds[-1] + 1 + max(0, n - len(seeds))))
    for s in seeds[:n]:
        if s not in _STACK:
            p = gen.draw_layer(dims, s)
            _STACK[s] = (p, q.DeviceLayer(p, G.dev()))
    return [_STACK[s][0] for s in seeds[:n]], [_STACK[s][1] for s in seeds[:n]]


@pytest.mark.parametrize("T", [1, 4])
def test_stack_40_layers(T):
    dims = gen.QWEN
    planes, layers = stack_layers(40)
    r0 = gen.draw_tokens(dims, T, 1000 + T, "resid")
    rref, recs = oracle.stack_forward(dims, planes, r0)
    ws = q.make_workspace(dims, T, G.dev())
    # with the oracle's routing forced at every layer
    resid = G.f32(r0)
    for li, dl in enumerate(layers):
        q.moe_block_forward(dims, dl, resid, ws, eps=1e-6, ids=G.i32(recs[li]["ids"]),
                            weights=G.f32(recs[li]["w"]))
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    G.assert_close(resid.cpu().numpy() - r0, rref - r0, f"40-layer stack T={T}, forced")
    # own routing: a token's ids are compared layer by layer while every
    # earlier layer kept it clear of a near tie (its residual then still
    # follows the oracle's)
    resid = G.f32(r0)
    ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=G.dev())
    x_out = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
    aligned = set(range(T))
    compared = 0
    for li, dl in enumerate(layers):
        q.moe_block_forward(dims, dl, resid, ws, eps=1e-6, x_out=x_out)
        q.moe_route(dims, dl, x_out, ids, torch.empty((T, dims.top_k), device=G.dev()),
                    torch.empty((T,), device=G.dev()), ws)
        torch.cuda.synchronize()
        got = ids.cpu().numpy()
        # the residuals differ by ~1e-3 relative after many layers: a gap of
        # 3e-3 keeps three times that margin
        clear = {t for t in aligned if recs[li]["gap"][t] >= 3e-3}
        for t in clear:
            assert np.array_equal(got[t], recs[li]["ids"][t]), (li, t)
            compared += 1
        aligned = clear
    assert compared >= 5, compared


@pytest.mark.parametrize("T", [1, 4])
def test_stack_40_layers_stack_call(T):
    """The 40-layer stack as the bench times it: one moe_stack_forward call,
    with the oracle's routing forced at every layer, and routed by itself over
    the leading layers free of near ties."""
    dims = gen.QWEN
    planes, layers = stack_layers(40)
    r0 = gen.draw_tokens(dims, T, 1000 + T, "resid")
    rref, recs = oracle.stack_forward(dims, planes, r0)
    ids = np.stack([rec["ids"] for rec in recs]).astype(np.int32)
    w = np.stack([rec["w"] for rec in recs]).astype(np.float32)
    ws = q.make_workspace(dims, T, G.dev())
    resid = G.f32(r0)
    q.moe_stack_forward(dims, layers, resid, ws, eps=1e-6, ids=G.i32(ids), weights=G.f32(w))
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    G.assert_close(resid.cpu().numpy() - r0, rref - r0, f"40-layer stack T={T}, stack call")
    # own routing: a token whose top-K gap stays clear (>= 3e-3) over its
    # leading layers routes there as the oracle does.  Over the longest such
    # run of any token (capped at 8 layers, at least one by the seeds), the
    # stack call with its own routing must then match, on those tokens, the
    # same call with the oracle's ids and weights forced.  The two differ by
    # the weights alone: the forced ones come from the oracle's logits, the
    # own ones from the kernels' (whose residual drifts ~1e-3 relative from
    # the oracle's along the stack), measured at 3.1e-3 relative after 8
    # layers of the tcgen05 path.  One expert chosen differently moves a row
    # by several percent, so a 1e-2 bar separates the two.  Tokens are
    # independent, so the others are free to differ.
    n_tok = G.leading_clear_layers(recs, 3e-3)
    n_ok = min(int(n_tok.max()), 8)
    assert n_ok >= 1, "every token meets a near tie in the first layer: pick another seed"
    rows = [t for t in range(T) if n_tok[t] >= n_ok]
    own = G.f32(r0)
    q.moe_stack_forward(dims, layers[:n_ok], own, ws, eps=1e-6)
    forced = G.f32(r0)
    q.moe_stack_forward(dims, layers[:n_ok], forced, ws, eps=1e-6, ids=G.i32(ids[:n_ok]),
                        weights=G.f32(w[:n_ok]))
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    d_own = own.cpu().numpy()[rows] - r0[rows]
    d_forced = forced.cpu().numpy()[rows] - r0[rows]
    rel = float(np.linalg.norm(d_own - d_forced) / np.linalg.norm(d_forced))
    assert rel <= 1e-2, f"{n_ok} layers, tokens {rows}: own routing off forced by {rel:.2e}"

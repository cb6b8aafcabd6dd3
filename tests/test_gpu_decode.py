"""Parity of decode-size layers (T <= 32) against the CPU oracle, through the
C ABI: the whole-layer calls (decode kernels up to
moe_layer_decode_max_tokens(), tcgen05 kernels above when the shape allows)
and the decode kernels themselves at every T through the stage calls.  Ids
and permutations bit-exact (near ties excepted, see gpu_util); floats within
rel-L2 5e-3 and max-abs 2e-2 * rms(ref)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_fwd_gb300 as q
from tests import gpu_util as G
from workloads import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    q.build.build()
    return q.load()


_LAYERS = {}


def layer(dims, seed, bias="none", alpha=0.0):
    key = (dims, seed, bias, alpha)
    if key not in _LAYERS:
        planes = gen.draw_layer(dims, seed, bias=bias, alpha=alpha)
        _LAYERS[key] = (planes, q.DeviceLayer(planes, G.dev()))
    return _LAYERS[key]


def qwen_x(T, seed, kind="resid"):
    r = gen.draw_tokens(gen.QWEN, T, seed, kind)
    return oracle.rmsnorm(r)


def gpu_layer(dims, dl, xb, forced=None):
    T = xb.shape[0]
    x = G.u16(xb)
    out = torch.full((T, dims.hidden), -1, dtype=torch.int16, device=G.dev())  # NaN sentinel
    ws = q.make_workspace(dims, T, G.dev())
    res = {}
    if forced is None:
        ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=G.dev())
        w = torch.empty((T, dims.top_k), dtype=torch.float32, device=G.dev())
        sig = torch.empty((T,), dtype=torch.float32, device=G.dev())
        q.moe_layer_forward(dims, dl, x, out, ws, ids=ids, weights=w, shared_gate=sig)
        res.update(ids=ids.cpu().numpy(), w=w.cpu().numpy(), sig=sig.cpu().numpy())
    else:
        q.moe_layer_forward_routed(dims, dl, x, G.i32(forced[0]), G.f32(forced[1]), out, ws)
    torch.cuda.synchronize()
    res["where"] = ws[:32].cpu().numpy().view(np.uint32)[1:8].tolist()
    res["status"] = q.moe_get_device_status(ws)
    res["out"] = G.bf16_to_np(out)
    return res


def check_layer(dims, planes, dl, xb, what):
    ref = oracle.moe_forward(dims, planes, xb)
    got = gpu_layer(dims, dl, xb)
    assert got["status"] == q.STRATA_OK, (what, got["status"], got["where"])
    clear = G.clear_tokens(ref["gap"])
    for t in clear:
        assert np.array_equal(got["ids"][t], ref["ids"][t]), (what, t)
        assert np.allclose(got["w"][t], ref["w"][t], rtol=1e-4, atol=1e-6), (what, t)
    assert np.allclose(got["sig"], ref["sig"], rtol=1e-4, atol=1e-6)
    if len(clear) == xb.shape[0]:
        G.assert_close(got["out"], ref["out"], what)
    else:
        G.assert_close(got["out"][clear], ref["out"][clear], what + " (clear tokens)")
        # near-tie tokens: floats checked with the oracle's routing forced
        forced = gpu_layer(dims, dl, xb, forced=(ref["ids"], ref["w"]))
        G.assert_close(forced["out"], ref["out"], what + " (forced)")
    return ref, got


def test_toy_layer(lib):
    dims = gen.TOY
    planes, dl = layer(dims, 0)
    xb = gen.draw_tokens(dims, 4, 0, "bf16")
    check_layer(dims, planes, dl, xb, "toy T=4")


@pytest.mark.parametrize("seed", range(10))
def test_decode1_qwen_layer(lib, seed):
    dims = gen.QWEN
    planes, dl = layer(dims, seed)
    check_layer(dims, planes, dl, qwen_x(1, seed), f"decode T=1 seed {seed}")


def test_decode16_pairs_zipf(lib):
    cfg = gen.CONFIGS["decode16"]
    dims = cfg.dims
    planes, dl = layer(dims, 0, bias="zipf", alpha=cfg.alpha)
    xb = qwen_x(16, 0, "pairs")
    ref, got = check_layer(dims, planes, dl, xb, "decode T=16")
    # the bucketing the fused kernel made equals the oracle's on the GPU's ids
    ids = G.i32(got["ids"])
    ws = q.make_workspace(dims, 16, G.dev())
    E, TK = dims.n_experts, 16 * dims.top_k
    counts = torch.empty(E, dtype=torch.int32, device=G.dev())
    offsets = torch.empty(E + 1, dtype=torch.int32, device=G.dev())
    perm = torch.empty(TK, dtype=torch.int32, device=G.dev())
    inv = torch.empty(TK, dtype=torch.int32, device=G.dev())
    q.moe_permute(dims, ids, counts, offsets, perm, inv, ws)
    oc, oo, op, oi = oracle.permute(got["ids"], E)
    assert np.array_equal(counts.cpu().numpy(), oc)
    assert np.array_equal(offsets.cpu().numpy(), oo)
    assert np.array_equal(perm.cpu().numpy(), op)
    assert np.array_equal(inv.cpu().numpy(), oi)


@pytest.mark.parametrize("T", [1, 2, 3, 7, 16, 31, 32])
def test_forced_routing_ragged_T(lib, T):
    dims = gen.QWEN
    planes, dl = layer(dims, 3)
    xb = qwen_x(T, 100 + T)
    ids, w = gen.draw_ids(T, dims.n_experts, dims.top_k, T)
    ref = oracle.moe_forward(dims, planes, xb, ids=ids, w=w)
    got = gpu_layer(dims, dl, xb, forced=(ids, w))
    assert got["status"] == q.STRATA_OK
    G.assert_close(got["out"], ref["out"], f"forced T={T}")


@pytest.mark.parametrize("T", [1, 5, 32])
def test_toy_ragged_T_routed(lib, T):
    dims = gen.TOY
    planes, dl = layer(dims, 7)
    xb = gen.draw_tokens(dims, T, 7 + T, "bf16")
    check_layer(dims, planes, dl, xb, f"toy T={T}")


def test_all_tokens_on_the_same_experts(lib):
    dims = gen.QWEN
    planes, dl = layer(dims, 4)
    T = 32
    xb = qwen_x(T, 44)
    ids = np.tile(np.arange(0, 8 * 31, 31, dtype=np.int32), (T, 1))
    w = np.full((T, dims.top_k), 0.125, dtype=np.float32)
    ref = oracle.moe_forward(dims, planes, xb, ids=ids, w=w)
    got = gpu_layer(dims, dl, xb, forced=(ids, w))
    G.assert_close(got["out"], ref["out"], "all tokens on 8 experts")


@pytest.mark.parametrize("E,K,I", [(4, 4, 64), (32, 1, 256), (16, 16, 1024)])
def test_degenerate_shapes(lib, E, K, I):
    dims = gen.LayerDims(hidden=512, n_experts=E, top_k=K, inter=I, shared_inter=128)
    planes, dl = layer(dims, 11)
    xb = gen.draw_tokens(dims, 6, 11, "bf16")
    check_layer(dims, planes, dl, xb, f"E={E} K={K} I={I}")


def test_hidden_1024_and_3072(lib):
    for H in (1024, 3072):
        dims = gen.LayerDims(hidden=H, n_experts=64, top_k=6, inter=256, shared_inter=512)
        planes, dl = layer(dims, 12)
        xb = gen.draw_tokens(dims, 5, 12, "bf16")
        check_layer(dims, planes, dl, xb, f"H={H}")


def test_separate_calls(lib):
    """route -> permute -> expert_ffn -> combine, each against the oracle."""
    dims = gen.QWEN
    planes, dl = layer(dims, 5)
    T, K, E, I = 6, dims.top_k, dims.n_experts, dims.inter
    xb = qwen_x(T, 55)
    ref = oracle.moe_forward(dims, planes, xb, want_y=True, want_h=True)
    x = G.u16(xb)
    ws = q.make_workspace(dims, T, G.dev())
    ids = torch.empty((T, K), dtype=torch.int32, device=G.dev())
    w = torch.empty((T, K), dtype=torch.float32, device=G.dev())
    sig = torch.empty((T,), dtype=torch.float32, device=G.dev())
    logits = torch.empty((T, E), dtype=torch.float32, device=G.dev())
    q.moe_route(dims, dl, x, ids, w, sig, ws, logits=logits)
    torch.cuda.synchronize()
    assert np.allclose(logits.cpu().numpy(), ref["logits"], rtol=0, atol=2e-5)
    clear = G.clear_tokens(ref["gap"])
    assert len(clear) == T
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    # continue with the oracle's routing so every later stage sees the same input
    ids = G.i32(ref["ids"])
    w = G.f32(ref["w"])
    counts = torch.empty(E, dtype=torch.int32, device=G.dev())
    offsets = torch.empty(E + 1, dtype=torch.int32, device=G.dev())
    perm = torch.empty(T * K, dtype=torch.int32, device=G.dev())
    inv = torch.empty(T * K, dtype=torch.int32, device=G.dev())
    q.moe_permute(dims, ids, counts, offsets, perm, inv, ws)
    oc, oo, op, oi = oracle.permute(ref["ids"], E)
    assert np.array_equal(perm.cpu().numpy(), op) and np.array_equal(inv.cpu().numpy(), oi)
    h = torch.empty((T * K, I), dtype=torch.float32, device=G.dev())
    q.moe_expert_gate_up(dims, dl, x, offsets, perm, h, ws)
    href = ref["h"].reshape(T * K, I)[op]
    G.assert_close(h.cpu().numpy(), href, "gate/up h", dtype="f32")
    y = torch.empty((T * K, dims.hidden), dtype=torch.int16, device=G.dev())
    q.moe_expert_ffn(dims, dl, x, offsets, perm, y, ws)
    yref = ref["y"].reshape(T * K, dims.hidden)[op]
    G.assert_close(G.bf16_to_np(y), yref, "expert y")
    y2 = torch.empty_like(y)
    q.moe_expert_down(dims, dl, h, T, offsets, y2, ws)
    assert torch.equal(y, y2)
    out = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
    q.moe_combine(dims, dl, x, y, inv, w, G.f32(ref["sig"]), out, ws)
    torch.cuda.synchronize()
    G.assert_close(G.bf16_to_np(out), ref["out"], "combine")
    assert q.moe_get_device_status(ws) == q.STRATA_OK


def test_bad_forced_id_latches_status(lib):
    dims = gen.TOY
    planes, dl = layer(dims, 0)
    xb = gen.draw_tokens(dims, 2, 3, "bf16")
    ids = np.array([[0, 1, 2, 3], [4, 5, 6, 99]], dtype=np.int32)
    w = np.full((2, 4), 0.25, dtype=np.float32)
    got = gpu_layer(dims, dl, xb, forced=(ids, w))
    assert got["status"] == q.STRATA_EBADROUTE
    # the token whose ids are all valid is still right
    ref = oracle.moe_forward(dims, planes, xb[:1], ids=ids[:1], w=w[:1])
    G.assert_close(got["out"][:1], ref["out"], "valid token beside a bad id")
    assert np.all(np.isfinite(got["out"]))


def test_zero_tokens_is_a_noop(lib):
    dims = gen.TOY
    _, dl = layer(dims, 0)
    x = torch.empty((0, dims.hidden), dtype=torch.int16, device=G.dev())
    out = torch.empty((0, dims.hidden), dtype=torch.int16, device=G.dev())
    ws = q.make_workspace(dims, 1, G.dev())
    q.moe_layer_forward(dims, dl, x, out, ws)
    assert q.moe_get_device_status(ws) == q.STRATA_OK


def test_unsupported_and_invalid_sizes(lib):
    dims = gen.TOY
    _, dl = layer(dims, 0)
    T = 8
    x = torch.zeros((T, dims.hidden), dtype=torch.int16, device=G.dev())
    out = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
    ws_small = q.make_workspace(dims, 2, G.dev())
    with pytest.raises(q.StrataError) as ei:
        q.moe_layer_forward(dims, dl, x, out, ws_small)
    assert ei.value.status == q.STRATA_EINVAL


def test_deterministic(lib):
    dims = gen.QWEN
    planes, dl = layer(dims, 6)
    xb = qwen_x(16, 66, "pairs")
    a = gpu_layer(dims, dl, xb)
    b = gpu_layer(dims, dl, xb)
    assert np.array_equal(a["out"].view(np.uint32), b["out"].view(np.uint32))
    assert np.array_equal(a["ids"], b["ids"])


def test_rmsnorm(lib):
    rng = np.random.default_rng(5)
    r = rng.normal(0, 2, (7, 2048)).astype(np.float32)
    x = torch.empty((7, 2048), dtype=torch.int16, device=G.dev())
    q.moe_rmsnorm(G.f32(r), x)
    torch.cuda.synchronize()
    got = x.cpu().numpy().view(np.uint16)
    want = oracle.rmsnorm(r)
    diff = np.abs(got.astype(np.int32) - want.astype(np.int32))
    # fp32 sums in another order: at most one bf16 ulp, on a handful of elements
    assert diff.max() <= 1 and (diff > 0).mean() < 1e-3


def test_block_forward_stack(lib):
    """Four residual blocks: with the oracle's routing forced at every block
    the final residual stays within tolerance of the oracle's."""
    dims = gen.QWEN
    layers = [layer(dims, 20 + i) for i in range(4)]
    T = 4
    r0 = gen.draw_tokens(dims, T, 9, "resid")
    rref, recs = oracle.stack_forward(dims, [p for p, _ in layers], r0)
    resid = G.f32(r0)
    ws = q.make_workspace(dims, T, G.dev())
    for li, (_, dl) in enumerate(layers):
        q.moe_block_forward(dims, dl, resid, ws, eps=1e-6, ids=G.i32(recs[li]["ids"]),
                            weights=G.f32(recs[li]["w"]))
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    G.assert_close(resid.cpu().numpy(), rref, "4-block stack, forced routing")
    # free-running: a token that meets no near tie in any block routes as the
    # oracle does and ends within tolerance of it (tokens are independent);
    # the seeds give at least one such token
    n_tok = G.leading_clear_layers(recs, 1e-3)
    rows = [t for t in range(T) if n_tok[t] == len(layers)]
    assert rows, "every token meets a near tie: pick other seeds"
    resid = G.f32(r0)
    for li, (_, dl) in enumerate(layers):
        x_out = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
        q.moe_block_forward(dims, dl, resid, ws, eps=1e-6, x_out=x_out)
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    G.assert_close(resid.cpu().numpy()[rows], rref[rows], f"4-block stack, own routing, {rows}")


def _static(lib, dims, dl, x, out, ids=None):
    d = q.dims_struct(dims)
    return lib.moe_layer_forward_static(ctypes.byref(d), ctypes.byref(dl.ptrs),
                                        ctypes.c_void_p(x.data_ptr()), x.shape[0],
                                        None if ids is None else ctypes.c_void_p(ids.data_ptr()),
                                        None, None, ctypes.c_void_p(out.data_ptr()), None)


def _stage_calls(dims, dl, x, ws, forced=None, ids=None):
    T = x.shape[0]
    out = torch.full((T, dims.hidden), -1, dtype=torch.int16, device=G.dev())
    if forced is None:
        q.moe_decode_route(dims, dl, x, ws)
        q.moe_decode_gate_up(dims, dl, x, ws, ids=ids)
    else:
        q.moe_decode_route(dims, dl, x, ws, forced=True)
        q.moe_decode_gate_up(dims, dl, x, ws, forced_ids=G.i32(forced[0]),
                             forced_weights=G.f32(forced[1]), ids=ids)
    q.moe_decode_down_combine(dims, dl, T, out, ws)
    return out


def test_stage_calls_equal_static_layer(lib):
    """moe_decode_route -> moe_decode_gate_up -> moe_decode_down_combine is
    the decode-kernel layer (moe_layer_forward_static), bit for bit, and
    publishes the same routing; where moe_layer_forward takes the persistent
    kernel (or the decode kernels), it is that layer too."""
    dims = gen.QWEN
    planes, dl = layer(dims, 8)
    for T in (1, 9):
        xb = qwen_x(T, 80 + T)
        x = G.u16(xb)
        out_a = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
        ids_a = torch.empty((T, dims.top_k), dtype=torch.int32, device=G.dev())
        assert _static(lib, dims, dl, x, out_a, ids_a) == q.STRATA_OK
        ids_b = torch.empty_like(ids_a)
        ws2 = q.make_workspace(dims, T, G.dev())
        out_b = _stage_calls(dims, dl, x, ws2, ids=ids_b)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b) and torch.equal(ids_a, ids_b)
        assert q.moe_get_device_status(ws2) == q.STRATA_OK
        if q.moe_layer_path(dims, T) in (q.PATH_PERSISTENT, q.PATH_DECODE):
            out_c = torch.empty_like(out_a)
            q.moe_layer_forward(dims, dl, x, out_c, ws2)
            torch.cuda.synchronize()
            assert torch.equal(out_a, out_c)


@pytest.mark.parametrize("T", [3, 7, 16, 31, 32])
def test_decode_kernels_ragged_T(lib, T):
    """The decode kernels above the whole-layer switch (the stage calls run
    them up to moe_decode_max_tokens()): ids on clear tokens, and the output
    with the oracle's routing forced, against the oracle."""
    dims = gen.QWEN
    planes, dl = layer(dims, 11)
    xb = qwen_x(T, 500 + T)
    ref = oracle.moe_forward(dims, planes, xb)
    ws = q.make_workspace(dims, T, G.dev())
    ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=G.dev())
    _stage_calls(dims, dl, G.u16(xb), ws, ids=ids)
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    got = ids.cpu().numpy()
    for t in G.clear_tokens(ref["gap"]):
        assert np.array_equal(got[t], ref["ids"][t]), t
    out = _stage_calls(dims, dl, G.u16(xb), ws, forced=(ref["ids"], ref["w"]))
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    G.assert_close(G.bf16_to_np(out), ref["out"], f"decode kernels T={T}")


def _oracle_stack_forced(dims, planes, r0):
    """The oracle's stack with its own routing, and the routing as arrays."""
    rref, recs = oracle.stack_forward(dims, planes, r0)
    ids = np.stack([rec["ids"] for rec in recs]).astype(np.int32)
    w = np.stack([rec["w"] for rec in recs]).astype(np.float32)
    return rref, recs, ids, w


@pytest.mark.parametrize("T", [1, 4, 16])
def test_stack_call_forced(lib, T):
    """moe_stack_forward with the oracle's routing forced at every layer: the
    final residual within tolerance of the oracle's; the last layer's output
    too."""
    dims = gen.QWEN
    layers = [layer(dims, 20 + i) for i in range(4)]
    planes = [p for p, _ in layers]
    r0 = gen.draw_tokens(dims, T, 90 + T, "resid")
    rref, recs, ids, w = _oracle_stack_forced(dims, planes, r0)
    resid = G.f32(r0)
    out = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
    ws = q.make_workspace(dims, T, G.dev())
    q.moe_stack_forward(dims, [dl for _, dl in layers], resid, ws, eps=1e-6, ids=G.i32(ids),
                        weights=G.f32(w), out=out)
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    G.assert_close(resid.cpu().numpy() - r0, rref - r0, f"4-layer stack T={T}, forced")
    G.assert_close(G.bf16_to_np(out), oracle.bf16_array_to_f32(recs[-1]["out_bf16"]),
                   "last layer's output")


def test_stack_call_own_routing(lib):
    """Routed by the kernel: ids agree with the oracle's, and the residual
    follows it, over the leading layers in which no token met a near tie."""
    dims = gen.QWEN
    layers = [layer(dims, 20 + i) for i in range(4)]
    planes = [p for p, _ in layers]
    T = 4
    r0 = gen.draw_tokens(dims, T, 9, "resid")
    rref, recs = oracle.stack_forward(dims, planes, r0)
    n_ok = 0
    while n_ok < len(recs) and np.all(recs[n_ok]["gap"] >= 3e-3):
        n_ok += 1
    assert n_ok >= 1, "pick another seed: the first layer already has a near tie"
    resid = G.f32(r0)
    ws = q.make_workspace(dims, T, G.dev())
    q.moe_stack_forward(dims, [dl for _, dl in layers[:n_ok]], resid, ws, eps=1e-6)
    torch.cuda.synchronize()
    assert q.moe_get_device_status(ws) == q.STRATA_OK
    want = r0 + sum(oracle.bf16_array_to_f32(recs[i]["out_bf16"]) for i in range(n_ok))
    G.assert_close(resid.cpu().numpy() - r0, want - r0, f"{n_ok}-layer stack, own routing")


def test_layer_profile_kernels(lib):
    """moe_layer_profile names the kernels of the path moe_layer_path reports:
    one persistent kernel at decode sizes, the tcgen05 kernels above (the
    bucketing fused into one kernel at T <= 32)."""
    dims = gen.QWEN
    _, dl = layer(dims, 0)
    want = {q.PATH_PERSISTENT: lambda T: q.PROFILE_PERSISTENT,
            q.PATH_DECODE: lambda T: q.PROFILE_DECODE,
            q.PATH_TC: lambda T: q.PROFILE_PREFILL_SMALL if T <= 32 else q.PROFILE_PREFILL}
    assert q.moe_layer_path(dims, 1) == q.PATH_PERSISTENT
    assert q.moe_layer_path(dims, 64) == q.PATH_TC
    for T in (1, 16, 24, 64):
        xt = qwen_x(T, 4)
        wst = q.make_workspace(dims, T, G.dev())
        ot = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
        prof = q.moe_layer_profile(dims, dl, G.u16(xt), ot, wst)
        assert list(prof) == list(want[q.moe_layer_path(dims, T)](T)), T
        assert all(v > 0 for v in prof.values())

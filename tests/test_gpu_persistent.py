"""The persistent decode kernel (one launch a layer, or a stack of layers)
through the C ABI.

It computes every step with the arithmetic of the three decode kernels, so
its results are compared with theirs BIT FOR BIT (the stage calls
moe_decode_route -> moe_decode_gate_up -> moe_decode_down_combine, and
moe_rmsnorm for a stack), besides the oracle comparisons of the other GPU
tests, which run through it wherever moe_layer_path says so.  Also: the
bucketing the layer's own kernels build (any path) bit-exact against the
oracle's stable sort, exact ties in the router broken by the lower id, the
grid-barrier flags across many calls and T values on one workspace, and a
grid barrier that runs out (bounded wait, latched STRATA_ETIMEOUT)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_fwd_gb300 as q
from tests import gpu_util as G
from workloads import gen

pytestmark = pytest.mark.gpu

_LAYERS = {}


@pytest.fixture(scope="module")
def lib():
    q.build.build()
    return q.load()


def layer(dims, seed, bias="none", alpha=0.0, planes=None):
    key = (dims, seed, bias, alpha)
    if planes is not None:
        return planes, q.DeviceLayer(planes, G.dev())
    if key not in _LAYERS:
        p = gen.draw_layer(dims, seed, bias=bias, alpha=alpha)
        _LAYERS[key] = (p, q.DeviceLayer(p, G.dev()))
    return _LAYERS[key]


def qwen_x(T, seed, kind="resid"):
    return oracle.rmsnorm(gen.draw_tokens(gen.QWEN, T, seed, kind))


def zeros_i16(T, H):
    return torch.full((T, H), -1, dtype=torch.int16, device=G.dev())


def stage_layer(dims, dl, x, ws, forced=None, resid=None):
    """The layer on the three decode kernels (the stage calls)."""
    T = x.shape[0]
    out = zeros_i16(T, dims.hidden)
    ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=G.dev())
    if forced is None:
        q.moe_decode_route(dims, dl, x, ws)
        q.moe_decode_gate_up(dims, dl, x, ws, ids=ids)
    else:
        q.moe_decode_route(dims, dl, x, ws, forced=True)
        q.moe_decode_gate_up(dims, dl, x, ws, forced_ids=forced[0], forced_weights=forced[1],
                             ids=ids)
    q.moe_decode_down_combine(dims, dl, T, out, ws, resid=resid)
    return out, ids


def persistent_layer(dims, dl, x, ws, forced=None):
    T = x.shape[0]
    out = zeros_i16(T, dims.hidden)
    ids = torch.empty((T, dims.top_k), dtype=torch.int32, device=G.dev())
    w = torch.empty((T, dims.top_k), dtype=torch.float32, device=G.dev())
    sig = torch.empty((T,), dtype=torch.float32, device=G.dev())
    if forced is None:
        q.moe_layer_forward(dims, dl, x, out, ws, ids=ids, weights=w, shared_gate=sig)
    else:
        q.moe_layer_forward_routed(dims, dl, x, forced[0], forced[1], out, ws)
    return out, ids, w, sig


def status(ws):
    where = ws[:32].cpu().numpy().view(np.uint32)[1:8].tolist()
    return q.moe_get_device_status(ws), where


def test_only_one_token_takes_the_persistent_kernel(lib):
    dims = gen.QWEN
    assert q.moe_layer_path(dims, 1) == q.PATH_PERSISTENT
    assert q.moe_layer_path(dims, 1, forced=True) == q.PATH_PERSISTENT
    for T in (2, 3, 4, 16):
        assert q.moe_layer_path(dims, T) != q.PATH_PERSISTENT, T


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_layer_bit_identical_to_decode_kernels(lib, seed):
    dims = gen.QWEN
    T = 1
    assert q.moe_layer_path(dims, T) == q.PATH_PERSISTENT
    _, dl = layer(dims, 30 + seed)
    x = G.u16(qwen_x(T, 300 + seed))
    ws_a = q.make_workspace(dims, T, G.dev())
    ws_b = q.make_workspace(dims, T, G.dev())
    out_a, ids_a, _, _ = persistent_layer(dims, dl, x, ws_a)
    out_b, ids_b = stage_layer(dims, dl, x, ws_b)
    torch.cuda.synchronize()
    assert status(ws_a)[0] == q.STRATA_OK, status(ws_a)
    assert status(ws_b)[0] == q.STRATA_OK
    assert torch.equal(ids_a, ids_b)
    assert torch.equal(out_a, out_b), "persistent kernel differs from the decode kernels"
    # forced routing (the oracle's rule: any ids, any weights)
    ids, w = gen.draw_ids(T, dims.n_experts, dims.top_k, 7 + seed)
    f = (G.i32(ids), G.f32(w))
    out_c, _, _, _ = persistent_layer(dims, dl, x, ws_a, forced=f)
    out_d, _ = stage_layer(dims, dl, x, ws_b, forced=f)
    torch.cuda.synchronize()
    assert status(ws_a)[0] == q.STRATA_OK
    assert torch.equal(out_c, out_d)


def test_zipf_bias_bit_identical(lib):
    """One token through a layer with the Zipf(1.1) router bias (the bias
    moves the selection)."""
    cfg = gen.CONFIGS["decode16"]
    dims = cfg.dims
    _, dl = layer(dims, 0, bias="zipf", alpha=cfg.alpha)
    x = G.u16(qwen_x(1, 0))
    ws_a = q.make_workspace(dims, 1, G.dev())
    ws_b = q.make_workspace(dims, 1, G.dev())
    out_a, ids_a, _, _ = persistent_layer(dims, dl, x, ws_a)
    out_b, ids_b = stage_layer(dims, dl, x, ws_b)
    torch.cuda.synchronize()
    assert status(ws_a)[0] == q.STRATA_OK
    assert torch.equal(ids_a, ids_b) and torch.equal(out_a, out_b)


@pytest.mark.parametrize("dims", [gen.TOY,
                                  gen.LayerDims(hidden=1024, n_experts=64, top_k=6, inter=256,
                                                shared_inter=512),
                                  gen.LayerDims(hidden=512, n_experts=16, top_k=16, inter=1024,
                                                shared_inter=64),
                                  gen.LayerDims(hidden=2048, n_experts=512, top_k=10, inter=512,
                                                shared_inter=512)],
                         ids=["toy", "h1024", "k16_i1024_is64", "e512_k10"])
def test_other_shapes_bit_identical(lib, dims):
    T = 1
    if q.moe_layer_path(dims, T) != q.PATH_PERSISTENT:
        pytest.skip("the persistent kernel does not take this shape on this GPU")
    _, dl = layer(dims, 41)
    x = G.u16(gen.draw_tokens(dims, T, 41, "bf16"))
    ws_a = q.make_workspace(dims, T, G.dev())
    ws_b = q.make_workspace(dims, T, G.dev())
    out_a, ids_a, _, _ = persistent_layer(dims, dl, x, ws_a)
    out_b, ids_b = stage_layer(dims, dl, x, ws_b)
    torch.cuda.synchronize()
    assert status(ws_a)[0] == q.STRATA_OK
    assert torch.equal(ids_a, ids_b) and torch.equal(out_a, out_b)


@pytest.mark.parametrize("T", [1])
def test_stack_bit_identical_to_kernel_chain(lib, T):
    """moe_stack_forward as one persistent launch against the same layers as
    separate kernels: moe_rmsnorm, then the three decode stages with the
    residual add, layer after layer."""
    dims = gen.QWEN
    if q.moe_layer_path(dims, T) != q.PATH_PERSISTENT:
        pytest.skip(f"T={T}: the stack takes the other kernels")
    layers = [layer(dims, 50 + i)[1] for i in range(6)]
    r0 = G.f32(gen.draw_tokens(dims, T, 60 + T, "resid"))
    ra = r0.clone()
    out_a = zeros_i16(T, dims.hidden)
    ws_a = q.make_workspace(dims, T, G.dev())
    q.moe_stack_forward(dims, layers, ra, ws_a, eps=1e-6, out=out_a)
    rb = r0.clone()
    ws_b = q.make_workspace(dims, T, G.dev())
    x = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
    for dl in layers:
        q.moe_rmsnorm(rb, x, eps=1e-6)
        out_b, _ = stage_layer(dims, dl, x, ws_b, resid=rb)
    torch.cuda.synchronize()
    assert status(ws_a)[0] == q.STRATA_OK, status(ws_a)
    assert status(ws_b)[0] == q.STRATA_OK
    assert torch.equal(out_a, out_b)
    assert torch.equal(ra.view(torch.int32), rb.view(torch.int32))


def test_block_forward_bit_identical(lib):
    dims = gen.QWEN
    _, dl = layer(dims, 55)
    T = 1
    r0 = G.f32(gen.draw_tokens(dims, T, 77, "resid"))
    ra, rb = r0.clone(), r0.clone()
    xa = zeros_i16(T, dims.hidden)
    oa = zeros_i16(T, dims.hidden)
    ws_a = q.make_workspace(dims, T, G.dev())
    q.moe_block_forward(dims, dl, ra, ws_a, eps=1e-6, x_out=xa, out=oa)
    xb = torch.empty_like(xa)
    q.moe_rmsnorm(rb, xb, eps=1e-6)
    ws_b = q.make_workspace(dims, T, G.dev())
    ob, _ = stage_layer(dims, dl, xb, ws_b, resid=rb)
    torch.cuda.synchronize()
    assert status(ws_a)[0] == q.STRATA_OK
    assert torch.equal(xa, xb) and torch.equal(oa, ob)
    assert torch.equal(ra.view(torch.int32), rb.view(torch.int32))


def test_many_calls_and_sizes_on_one_workspace(lib):
    """The barrier flags live at a fixed place in the workspace and every
    launch leaves them equal: calls of different T (and a stack) in any
    order on one workspace keep giving the same bits."""
    dims = gen.QWEN
    _, dl = layer(dims, 31)
    ws = q.make_workspace(dims, 16, G.dev())
    xs = {T: G.u16(qwen_x(T, 900 + T)) for T in (1, 3, 4)}
    first = {}
    for rep in range(3):
        for T in (1, 4, 3, 1):
            out, _, _, _ = persistent_layer(dims, dl, xs[T], ws)
            if T not in first:
                first[T] = out.clone()
            else:
                assert torch.equal(out, first[T]), (rep, T)
        r = G.f32(gen.draw_tokens(dims, 2, 5, "resid"))
        q.moe_stack_forward(dims, [dl] * 3, r, ws, eps=1e-6)
    torch.cuda.synchronize()
    assert status(ws)[0] == q.STRATA_OK, status(ws)
    flags = ws[256:256 + 4 * 1024].cpu().numpy().view(np.uint32)   # exchange counters
    sms = torch.cuda.get_device_properties(G.dev()).multi_processor_count
    assert np.all(flags[:sms] == flags[0]) and flags[0] > 0 and np.all(flags[sms:] == 0)


def _bucketing(dims, T, ws):
    E, TK = dims.n_experts, T * dims.top_k
    c = torch.empty(E, dtype=torch.int32, device=G.dev())
    o = torch.empty(E + 1, dtype=torch.int32, device=G.dev())
    p = torch.empty(TK, dtype=torch.int32, device=G.dev())
    i = torch.empty(TK, dtype=torch.int32, device=G.dev())
    q.moe_layer_bucketing(dims, T, ws, c, o, p, i)
    return [a.cpu().numpy() for a in (c, o, p, i)]


@pytest.mark.parametrize("T", [1, 3, 16, 32, 33, 300, 2048])
def test_layer_bucketing_bit_exact(lib, T):
    """The bucketing the whole-layer call's own kernels built (persistent at
    decode sizes, the tcgen05 kernels' single-CTA sort up to 32 tokens and
    count / scan / scatter above) against the oracle's stable sort of the
    ids the call published; and those ids against the oracle's routing on
    every token away from a near tie."""
    cfg = gen.CONFIGS["prefill"]
    dims = cfg.dims
    planes, dl = layer(dims, 0, bias="zipf", alpha=cfg.alpha)
    xb = qwen_x(T, 2000 + T)
    ws = q.make_workspace(dims, T, G.dev())
    out, ids, _, _ = persistent_layer(dims, dl, G.u16(xb), ws)
    got = _bucketing(dims, T, ws)
    torch.cuda.synchronize()
    assert status(ws)[0] == q.STRATA_OK
    ids_np = ids.cpu().numpy()
    want = oracle.permute(ids_np, dims.n_experts)
    for g, w, name in zip(got, want, ("counts", "offsets", "perm", "inv")):
        assert np.array_equal(g, w), (T, name)
    if T <= 300:
        ref_logits, _ = oracle.router(xb, planes["router"], planes.get("router_bias"))
        ref_ids, _, gap = oracle.select(ref_logits, dims.top_k)
        for t in G.clear_tokens(gap):
            assert np.array_equal(ids_np[t], ref_ids[t]), t


def _tie_planes(dims, seed, mode):
    """A layer whose router gives exact ties: `zero`, every router row 0
    (all logits equal); `dup`, every row a copy of row 0 except four."""
    planes = dict(gen.draw_layer(dims, seed))
    r = np.array(planes["router"], copy=True).reshape(dims.n_experts + 1, dims.hidden)
    if mode == "zero":
        r[:dims.n_experts] = 0
    else:
        keep = r[[100, 101, 102, 103]].copy()
        r[:dims.n_experts] = r[0]
        r[[100, 101, 102, 103]] = keep
    planes["router"] = r.reshape(np.asarray(planes["router"]).shape)
    planes["router_bias"] = None
    return planes


@pytest.mark.parametrize("mode", ["zero", "dup"])
@pytest.mark.parametrize("T", [1, 16, 300])
def test_exact_ties_lower_id_wins(lib, mode, T):
    """Exact ties in the router (identical rows give identical fp32 sums)
    are compared bit-exactly, not set aside as near ties: the lower expert
    id wins (PolyStrata, "What was tuned": the first of equal values).  With
    every logit equal the ids are 0..K-1 and every weight 1/K."""
    dims = gen.QWEN
    planes = _tie_planes(dims, 70, mode)
    _, dl = layer(dims, None, planes=planes)
    xb = qwen_x(T, 3000 + T)
    ws = q.make_workspace(dims, T, G.dev())
    out, ids, w, _ = persistent_layer(dims, dl, G.u16(xb), ws)
    torch.cuda.synchronize()
    assert status(ws)[0] == q.STRATA_OK
    ref = oracle.moe_forward(dims, planes, xb)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"]), (mode, T)
    assert np.allclose(w.cpu().numpy(), ref["w"], rtol=1e-5, atol=1e-7)
    if mode == "zero":
        K = dims.top_k
        assert np.array_equal(ref["ids"], np.tile(np.arange(K, dtype=np.int32), (T, 1)))
        assert np.allclose(w.cpu().numpy(), 1.0 / K, rtol=1e-6)
    else:
        assert np.all(np.sum(ref["ids"] < 100, axis=1) >= dims.top_k - 4)
    G.assert_close(G.bf16_to_np(out), ref["out"], f"ties {mode} T={T}")
    if T <= q.moe_decode_max_tokens():
        # the three decode kernels break the ties the same way
        ws2 = q.make_workspace(dims, T, G.dev())
        _, ids2 = stage_layer(dims, dl, G.u16(xb), ws2)
        torch.cuda.synchronize()
        assert np.array_equal(ids2.cpu().numpy(), ref["ids"])


def test_wait_for_another_cta_runs_out(lib):
    """A wait for another CTA's data that never comes runs out, latches
    STRATA_ETIMEOUT, records the site and lets the kernel finish.  One CTA's
    exchange counter in the workspace is moved ahead, so the words it writes
    carry tags nobody waits for and it waits for tags nobody writes; the poll
    budget is cut so the wait ends in about a millisecond.  The context stays
    usable: with the counters made equal again (raised, never lowered: a
    lower tag could match a word an earlier launch left) the next call is
    right again."""
    dims = gen.QWEN
    _, dl = layer(dims, 32)
    T = 1
    assert q.moe_layer_path(dims, T) == q.PATH_PERSISTENT
    x = G.u16(qwen_x(T, 1234))
    ws = q.make_workspace(dims, T, G.dev())
    good, _, _, _ = persistent_layer(dims, dl, x, ws)
    torch.cuda.synchronize()
    assert status(ws)[0] == q.STRATA_OK
    flags = ws[256:256 + 4 * 1024].view(torch.int32)
    sms = torch.cuda.get_device_properties(G.dev()).multi_processor_count
    try:
        q.strata_set_grid_wait_limit(2000)
        flags[5] += 1000
        persistent_layer(dims, dl, x, ws)
        torch.cuda.synchronize()
        st, where = status(ws)
    finally:
        q.strata_set_grid_wait_limit(0)
    assert st == q.STRATA_ETIMEOUT
    assert where[0] in (80, 81, 82) and where[6] == 1, where
    flags[:sms] = flags[:sms].max() + 16
    again, _, _, _ = persistent_layer(dims, dl, x, ws)
    torch.cuda.synchronize()
    assert status(ws)[0] == q.STRATA_OK
    assert torch.equal(again, good)

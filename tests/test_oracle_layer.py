"""Pins of the oracle's expert FFN, combine and whole layer."""
import numpy as np
import pytest
import torch

import oracle
from tests import brute
from workloads import gen


def _rel_l2(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def test_expert_dense_against_float64():
    rng = np.random.default_rng(20)
    H, I = 256, 64
    x = rng.normal(0, 1, H).astype(np.float32)
    Wgu = (rng.normal(0, 0.1, (2 * I, H))).astype(np.float32)
    Wd = (rng.normal(0, 0.1, (H, I))).astype(np.float32)
    h, y = oracle.expert_dense(x, Wgu, Wd)
    hr, yr = brute.expert(x.astype(np.float64), Wgu.astype(np.float64), Wd.astype(np.float64))
    assert _rel_l2(h, hr) < 1e-5 and _rel_l2(y, yr) < 1e-5


def test_zero_gate_rows_give_zero_output():
    # silu(0) = 0: with every gate row zero the expert's output is exactly 0
    rng = np.random.default_rng(21)
    H, I = 128, 32
    x = rng.normal(0, 1, H).astype(np.float32)
    Wgu = rng.normal(0, 0.1, (2 * I, H)).astype(np.float32)
    Wgu[0::2] = 0.0
    Wd = rng.normal(0, 0.1, (H, I)).astype(np.float32)
    h, y = oracle.expert_dense(x, Wgu, Wd)
    assert np.all(h == 0.0) and np.all(y == 0.0)


def _zero_shared(L):
    L = dict(L)
    L["sh_gu_s"] = np.zeros_like(L["sh_gu_s"])
    L["sh_dn_s"] = np.zeros_like(L["sh_dn_s"])
    return L


def test_one_hot_routing_equals_single_dense_expert():
    """Forced ids with weights (1, 0, ...) and a zeroed shared expert: the
    layer equals one dense SwiGLU FFN, (silu(x Wg^T) * (x Wu^T)) Wd^T, done
    in float64 on the dequantised matrices."""
    dims = gen.TOY
    L = _zero_shared(gen.draw_layer(dims, 1))
    T, K = 3, dims.top_k
    x = gen.draw_tokens(dims, T, 1, "bf16")
    ids = np.array([[0, 5, 9, 30], [3, 4, 5, 6], [1, 2, 17, 31]], dtype=np.int32)
    w = np.zeros((T, K), dtype=np.float32)
    w[:, 0] = 1.0
    res = oracle.moe_forward(dims, L, x, ids=ids, w=w)
    xf = brute.bf16_bits_to_f64(x)
    H, I = dims.hidden, dims.inter
    for t in range(T):
        e = ids[t, 0]
        Wgu = brute.dequant_xor(L["gu_q"][e], L["gu_s"][e], 2 * I, H)
        Wd = brute.dequant_xor(L["dn_q"][e], L["dn_s"][e], H, I)
        g = Wgu[0::2] @ xf[t]
        u = Wgu[1::2] @ xf[t]
        ref = Wd @ ((g / (1 + np.exp(-g))) * u)
        assert _rel_l2(res["out"][t], ref) < 1e-5


def test_combine_linearity_and_order():
    dims = gen.TOY
    L = gen.draw_layer(dims, 2)
    T = 4
    x = gen.draw_tokens(dims, T, 2, "bf16")
    ids, w = gen.draw_ids(T, dims.n_experts, dims.top_k, 2)
    a = oracle.moe_forward(dims, L, x, ids=ids, w=w, want_shared=True)
    routed_a = a["out"] - a["sig"][:, None] * a["shared"]
    b = oracle.moe_forward(dims, L, x, ids=ids, w=2.5 * w, want_shared=True)
    routed_b = b["out"] - b["sig"][:, None] * b["shared"]
    assert _rel_l2(routed_b, 2.5 * routed_a) < 1e-6
    # swapping two ids together with their weights leaves the layer unchanged
    ids2, w2 = ids.copy(), w.copy()
    ids2[:, [0, 2]] = ids2[:, [2, 0]]
    w2[:, [0, 2]] = w2[:, [2, 0]]
    c = oracle.moe_forward(dims, L, x, ids=ids2, w=w2)
    assert _rel_l2(c["out"], a["out"]) < 1e-6


def test_shared_gate_is_sigmoid_of_gate_row():
    dims = gen.TOY
    L = gen.draw_layer(dims, 3)
    x = gen.draw_tokens(dims, 2, 3, "bf16")
    res = oracle.moe_forward(dims, L, x)
    s = brute.bf16_bits_to_f64(x) @ brute.bf16_bits_to_f64(L["router"])[dims.n_experts]
    assert np.allclose(res["sig"], 1 / (1 + np.exp(-s)), rtol=1e-5, atol=0)


@pytest.mark.parametrize("T", [1, 4])
def test_toy_layer_against_float64_brute_force(T):
    dims = gen.TOY
    L = gen.draw_layer(dims, 0)
    x = gen.draw_tokens(dims, T, 0, "bf16")
    res = oracle.moe_forward(dims, L, x)
    ref = brute.layer(dims, L, x)
    for t in range(T):
        assert ref["gap"][t] > 1e-4
        assert np.array_equal(res["ids"][t], ref["ids"][t])
    assert _rel_l2(res["out"], ref["out"]) < 1e-5


def test_qwen_layer_against_float64_brute_force_one_token():
    dims = gen.QWEN
    L = gen.draw_layer(dims, 0)
    r = gen.draw_tokens(dims, 1, 0, "resid")
    x = oracle.rmsnorm(r)
    res = oracle.moe_forward(dims, L, x)
    ref = brute.layer(dims, L, x)
    assert ref["gap"][0] > 1e-4
    assert np.array_equal(res["ids"][0], ref["ids"][0])
    assert _rel_l2(res["out"], ref["out"]) < 1e-5


def test_layer_with_bias_routes_on_biased_logits():
    dims = gen.TOY
    L = gen.draw_layer(dims, 4, bias="zipf", alpha=1.0)
    x = gen.draw_tokens(dims, 4, 4, "bf16")
    res = oracle.moe_forward(dims, L, x)
    ref = brute.layer(dims, L, x)
    for t in range(4):
        if ref["gap"][t] > 1e-4:
            assert np.array_equal(res["ids"][t], ref["ids"][t])
    assert _rel_l2(res["out"], ref["out"]) < 1e-5


def test_forced_bad_id_is_refused():
    dims = gen.TOY
    L = gen.draw_layer(dims, 0)
    x = gen.draw_tokens(dims, 1, 0, "bf16")
    with pytest.raises(ValueError):
        oracle.moe_forward(dims, L, x, ids=np.array([[0, 1, 2, 32]], dtype=np.int32),
                           w=np.ones((1, 4), dtype=np.float32))


def test_thread_count_does_not_change_bits():
    dims = gen.TOY
    L = gen.draw_layer(dims, 5)
    x = gen.draw_tokens(dims, 4, 5, "bf16")
    a = oracle.moe_forward(dims, L, x, nthreads=1)
    b = oracle.moe_forward(dims, L, x, nthreads=4)
    assert np.array_equal(a["out"], b["out"])


def test_rmsnorm_against_float64():
    rng = np.random.default_rng(22)
    r = rng.normal(0, 3, (4, 2048)).astype(np.float32)
    x = oracle.rmsnorm(r, 1e-6)
    rd = r.astype(np.float64)
    ref = rd / np.sqrt((rd * rd).mean(axis=1, keepdims=True) + 1e-6)
    xf = brute.bf16_bits_to_f64(x)
    # bf16 keeps 8 significant bits: within half an ulp plus fp32 noise
    assert np.all(np.abs(xf - ref) <= np.abs(ref) * (2.0 ** -8 + 1e-6) + 1e-30)
    # closed form: a constant row c normalises to c / sqrt(c^2 + eps)
    c = np.full((1, 64), 2.0, dtype=np.float32)
    xc = brute.bf16_bits_to_f64(oracle.rmsnorm(c, 1e-6))
    assert np.all(xc == 1.0)


def test_stack_residual_chain_two_layers():
    dims = gen.TOY
    layers = [gen.draw_layer(dims, s) for s in (0, 1)]
    r0 = gen.draw_tokens(dims, 2, 9, "resid")
    r, recs = oracle.stack_forward(dims, layers, r0)
    # replaying the chain step by step gives the same bits
    rr = r0.copy()
    for li, L in enumerate(layers):
        x = oracle.rmsnorm(rr)
        assert np.array_equal(x, recs[li]["x"])
        out = oracle.moe_forward(dims, L, x)["out"]
        rr = rr + oracle.bf16_array_to_f32(oracle.round_bf16(out))
    assert np.array_equal(r, rr)


def _bf16_bits_f64(a):
    """float64 -> bf16 bits, round to nearest even (torch's conversion)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _round_like(v, got_bits, tol):
    """Rounds the float64 values v to bf16 and checks the oracle's bits
    got_bits against them: a correct rounding of a value computed within
    `tol` (absolute, per element: the fp32 error bound) of v is a bf16 value
    within half a bf16 ulp of v plus tol.  Where the oracle's bits differ
    from v's own rounding but obey that bound, they are kept.  Returns the
    bits to continue with and the number of elements that broke the bound."""
    v = np.asarray(v, dtype=np.float64)
    want = _bf16_bits_f64(v)
    got = np.asarray(got_bits, dtype=np.uint16).reshape(v.shape)
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(v), 1e-300))) - 8.0)
    ok = (got == want) | (np.abs(brute.bf16_bits_to_f64(got) - v) <= half_ulp + tol)
    return np.where(ok, got, want), int((~ok).sum())


def _stack64(dims, layers, r0, recs, forced=None):
    """The residual stack in float64 with no oracle arithmetic: r +=
    bf16(layer(x)), x = bf16(r / sqrt(mean(r^2) + 1e-6)), each layer by the
    float64 brute force.  At each bf16 rounding the oracle's bits (recs) must
    be the float64 chain's, except within fp32 error of a rounding midpoint,
    where the oracle's choice of neighbour is followed.  Returns the final r
    and the number of roundings that broke that rule."""
    r = np.asarray(r0, dtype=np.float64).copy()
    bad = 0
    for li, L in enumerate(layers):
        xn = r / np.sqrt((r * r).mean(axis=1, keepdims=True) + 1e-6)
        xb, n = _round_like(xn, recs[li]["x"], 4e-7 * np.abs(xn) + 1e-30)
        bad += n
        if forced is None:
            res = brute.layer(dims, L, xb)
        else:
            res = brute.layer(dims, L, xb, ids=forced[li][0], w=forced[li][1])
        out = res["out"]
        rms = np.sqrt((out * out).mean(axis=1, keepdims=True))
        ob, n = _round_like(out, recs[li]["out_bf16"], 1e-5 * np.abs(out) + 1e-6 * rms)
        bad += n
        r = r + brute.bf16_bits_to_f64(ob)
    return r, bad


def test_stack_against_float64_composition():
    """stack_forward against the chain written out in float64 from the
    brute-force layer (no oracle function on the reference side): every
    rounded input and output of every layer is the float64 chain's (up to
    the choice of neighbour within fp32 error of a bf16 midpoint) and the
    final residual agrees to fp32 accumulation error."""
    dims = gen.TOY
    layers = [gen.draw_layer(dims, s) for s in (3, 4, 5)]
    r0 = gen.draw_tokens(dims, 3, 9, "resid")
    r, recs = oracle.stack_forward(dims, layers, r0)
    r64, bad = _stack64(dims, layers, r0, recs)
    assert bad == 0
    rel = np.linalg.norm(r - r64) / np.linalg.norm(r64)
    assert rel < 1e-6, rel
    # a misplaced rounding is far larger: leaving out the bf16 rounding of
    # each layer's output moves r by ~1e-4 relative
    r_noround = np.asarray(r0, dtype=np.float64).copy()
    for L in layers:
        xn = r_noround / np.sqrt((r_noround ** 2).mean(axis=1, keepdims=True) + 1e-6)
        r_noround = r_noround + brute.layer(dims, L, _bf16_bits_f64(xn))["out"]
    assert np.linalg.norm(r - r_noround) / np.linalg.norm(r64) > 20 * rel


def test_stack_one_hot_routing_two_layers():
    """Forced one-hot routing (weight 1 on one expert, 0 on the others) in a
    2-layer stack: each layer is the shared expert plus one dense SwiGLU FFN;
    stack_forward must follow the float64 chain."""
    dims = gen.TOY
    layers = [gen.draw_layer(dims, s) for s in (6, 7)]
    T, K = 2, dims.top_k
    r0 = gen.draw_tokens(dims, T, 11, "resid")
    forced = []
    for li in range(2):
        ids = np.array([[3 + li, 10, 20, 30], [0, 5 + li, 17, 31]], dtype=np.int32)[:, :K]
        w = np.zeros((T, K), dtype=np.float32)
        w[0, 0] = 1.0
        w[1, 1] = 1.0
        forced.append((ids, w))
    r, recs = oracle.stack_forward(dims, layers, r0, forced=forced)
    r64, bad = _stack64(dims, layers, r0, recs, forced=forced)
    assert bad == 0
    assert np.linalg.norm(r - r64) / np.linalg.norm(r64) < 1e-6

"""Pins of the oracle's expert FFN, combine and whole layer."""
import numpy as np
import pytest

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

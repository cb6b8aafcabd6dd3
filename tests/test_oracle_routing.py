"""Pins of the oracle's router, top-K selection, softmax and permutation."""
import itertools
import math

import numpy as np

import oracle
from tests import brute
from workloads import gen


def _beats(la, a, lb, b):
    return la > lb or (la == lb and a < b)


def test_router_against_float64_matmul():
    rng = np.random.default_rng(10)
    T, H, E = 3, 512, 32
    x = gen._bf16_bits(rng.normal(0, 1, (T, H)).astype(np.float32))
    R = gen._bf16_bits(rng.normal(0, 0.02, (E + 1, H)).astype(np.float32))
    bias = rng.normal(0, 1, E).astype(np.float32)
    logits, gate = oracle.router(x, R, bias)
    xf = brute.bf16_bits_to_f64(x)
    Rf = brute.bf16_bits_to_f64(R)
    ref = xf @ Rf[:E].T + bias
    # serial fp32 sum of n terms: |err| <= n * eps * sum |x_h w_h| (+ the bias add)
    bound = (H + 1) * 2.0 ** -24 * (np.abs(xf) @ np.abs(Rf[:E]).T + np.abs(bias))
    assert np.all(np.abs(logits - ref) <= bound)
    refg = xf @ Rf[E]
    assert np.all(np.abs(gate - refg) <= H * 2.0 ** -24 * (np.abs(xf) @ np.abs(Rf[E])))


def test_router_unit_rows_pick_single_inputs():
    # router row e = unit vector on input e: logit e is exactly x[e]
    T, H, E = 2, 64, 8
    rng = np.random.default_rng(11)
    x = gen._bf16_bits(rng.normal(0, 1, (T, H)).astype(np.float32))
    R = np.zeros((E + 1, H), dtype=np.uint16)
    for e in range(E):
        R[e, 3 * e] = 0x3F80                      # 1.0
    R[E, 5] = 0xC000                              # gate = -2 x[5]
    logits, gate = oracle.router(x, R, None)
    xf = brute.bf16_bits_to_f64(x)
    for e in range(E):
        assert np.all(logits[:, e] == xf[:, 3 * e].astype(np.float32))
    assert np.all(gate == (-2.0 * xf[:, 5]).astype(np.float32))


def test_select_all_equal_closed_form():
    for E, K in [(32, 4), (256, 8), (8, 8)]:
        ids, w, gap = oracle.select(np.zeros((2, E), dtype=np.float32), K)
        assert np.array_equal(ids, np.tile(np.arange(K, dtype=np.int32), (2, 1)))
        assert np.allclose(w, 1.0 / K, rtol=0, atol=1e-7)
        if K < E:
            assert np.all(gap == 0.0)
        else:
            assert np.all(np.isinf(gap))


def test_select_two_logits_closed_form():
    # logits ln 2 and 0 on the only two experts: weights 2/3 and 1/3
    l = np.array([[0.0, math.log(2.0), -5.0, -6.0]], dtype=np.float32)
    ids, w, gap = oracle.select(l, 2)
    assert list(ids[0]) == [0, 1]
    assert abs(w[0, 0] - 1.0 / 3.0) < 1e-6 and abs(w[0, 1] - 2.0 / 3.0) < 1e-6
    assert abs(gap[0] - 5.0) < 1e-6


def test_select_is_a_top_k_set_brute_force():
    """For every token the selected set beats every unselected expert, the ids
    ascend, and the set equals the one exhaustive search over all K-subsets
    finds (largest sum of logits; among equal sums the lexicographically
    smallest ids), checked on small E with many exact ties."""
    rng = np.random.default_rng(12)
    for E, K in [(6, 2), (7, 3), (8, 4), (9, 1)]:
        for _ in range(60):
            l = rng.integers(-3, 4, size=(1, E)).astype(np.float32)   # many ties
            ids, w, gap = oracle.select(l, K)
            sel = set(int(i) for i in ids[0])
            assert list(ids[0]) == sorted(ids[0]) and len(sel) == K
            for a in sel:
                for b in set(range(E)) - sel:
                    assert _beats(l[0, a], a, l[0, b], b)
            best = None
            for sub in itertools.combinations(range(E), K):
                key = (-sum(float(l[0, e]) for e in sub), sub)
                best = key if best is None or key < best else best
            assert tuple(int(i) for i in ids[0]) == best[1]


def test_softmax_invariants():
    rng = np.random.default_rng(13)
    l = rng.normal(0, 3, (50, 64)).astype(np.float32)
    ids, w, gap = oracle.select(l, 8)
    assert np.all(np.abs(w.sum(axis=1) - 1.0) <= 1e-6)
    for t in range(50):
        ls = l[t, ids[t]].astype(np.float64)
        # weight ratios follow exp of logit differences
        for a in range(8):
            for b in range(8):
                assert abs(w[t, a] / w[t, b] - math.exp(ls[a] - ls[b])) <= \
                    2e-6 * math.exp(ls[a] - ls[b])
        srt = np.sort(l[t].astype(np.float64))[::-1]
        assert abs(gap[t] - (srt[7] - srt[8])) <= 1e-6 * max(1.0, abs(srt[7]))


def test_select_agrees_with_float64_brute_force_layer_routing():
    dims = gen.TOY
    L = gen.draw_layer(dims, 0)
    x = gen.draw_tokens(dims, 8, 0, "bf16")
    logits, _ = oracle.router(x, L["router"], None)
    ids, w, gap = oracle.select(logits, dims.top_k)
    ref = brute.layer(dims, L, x)
    for t in range(8):
        if ref["gap"][t] > 1e-4:
            assert np.array_equal(ids[t], ref["ids"][t])
            assert np.allclose(w[t], ref["w"][t], rtol=2e-6, atol=1e-7)


def test_sigmoid_and_swiglu_closed_forms():
    assert oracle.sigmoid(0.0) == 0.5
    assert abs(oracle.sigmoid(math.log(3.0)) - 0.75) < 1e-7
    assert abs(oracle.sigmoid(-math.log(3.0)) - 0.25) < 1e-7
    assert oracle.swiglu(0.0, 5.0) == 0.0
    assert abs(oracle.swiglu(math.log(3.0), 2.0) - 2.0 * 0.75 * math.log(3.0)) < 1e-6
    assert abs(oracle.swiglu(30.0, 1.0) - 30.0) < 1e-5
    assert abs(oracle.swiglu(-30.0, 1.0)) < 1e-10


def test_permute_invariants():
    rng = np.random.default_rng(14)
    for T, E, K in [(1, 256, 8), (16, 256, 8), (37, 32, 4), (0, 8, 2), (5, 8, 8)]:
        ids = np.zeros((T, K), dtype=np.int32)
        for t in range(T):
            ids[t] = np.sort(rng.choice(E, K, replace=False))
        counts, offsets, perm, inv = oracle.permute(ids, E)
        assert offsets[0] == 0 and offsets[E] == T * K
        assert np.array_equal(counts, np.bincount(ids.ravel(), minlength=E))
        assert np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(perm[inv], np.arange(T * K))
        assert np.array_equal(inv[perm], np.arange(T * K))
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(ids.ravel()[seg] == e)
            assert np.all(np.diff(seg // K) > 0)           # ascending tokens


def test_permute_all_tokens_to_one_expert():
    T, K, E = 9, 1, 4
    ids = np.full((T, K), 2, dtype=np.int32)
    counts, offsets, perm, inv = oracle.permute(ids, E)
    assert list(counts) == [0, 0, 9, 0]
    assert list(offsets) == [0, 0, 0, 9, 9]
    assert list(perm) == list(range(9)) and list(inv) == list(range(9))

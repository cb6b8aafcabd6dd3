"""Pins of the oracle's tail-skip (PolyStrata, "Models and backends", section
"What was tuned": an expert that every token of a call ranks at place n + 1
or later of its picks is left out; the picks that stay keep their weights).
Each pin would fail for a plausible mistake: ranking the wrong way round,
skipping per token instead of per call, renormalising the kept weights,
an off-by-one in the place, or ties broken towards the higher id."""
import numpy as np
import pytest

import oracle
from workloads import gen


def test_hand_computed_two_tokens():
    # token 0 ranks 1, 3, 5, 7 in that order, token 1 ranks 9, 5, 3, 2; with
    # n = 2 the kept experts are {1, 3} and {9, 5}: 7 and 2 go, 5 stays
    # because token 1 places it second although token 0 places it third
    ids = np.array([[1, 3, 5, 7], [2, 3, 5, 9]])
    w = np.array([[0.4, 0.3, 0.2, 0.1], [0.1, 0.2, 0.3, 0.4]], dtype=np.float32)
    w2, sk = oracle.tail_skip(ids, w, 2)
    assert sk.tolist() == [[False, False, False, True], [True, False, False, False]]
    np.testing.assert_array_equal(
        w2, np.array([[0.4, 0.3, 0.2, 0.0], [0.0, 0.2, 0.3, 0.4]], dtype=np.float32))


def test_tie_goes_to_the_lower_id():
    # equal weights: the lower id takes the better place, so with n = 1 of a
    # single token the lower id stays
    ids = np.array([[4, 9]])
    w = np.array([[0.5, 0.5]], dtype=np.float32)
    _, sk = oracle.tail_skip(ids, w, 1)
    assert sk.tolist() == [[False, True]]


@pytest.mark.parametrize("n", [0, 8, 9])
def test_off_leaves_every_pick(n):
    rng = np.random.default_rng(1)
    ids = np.stack([np.sort(rng.choice(64, 8, replace=False)) for _ in range(5)])
    w = rng.random((5, 8)).astype(np.float32)
    w2, sk = oracle.tail_skip(ids, w, n)
    assert not sk.any()
    assert np.array_equal(w2, w)


@pytest.mark.parametrize("n", [1, 3, 5, 7])
def test_single_token_drops_its_lowest(n):
    # one token: the K - n picks of lowest weight (ties: higher id last) go
    rng = np.random.default_rng(n)
    K = 8
    ids = np.sort(rng.choice(256, K, replace=False))[None, :]
    w = rng.random((1, K)).astype(np.float32)
    order = np.lexsort((ids[0], -w[0]))            # best first
    want = np.zeros(K, dtype=bool)
    want[order[n:]] = True
    w2, sk = oracle.tail_skip(ids, w, n)
    assert np.array_equal(sk[0], want)
    assert np.array_equal(w2[0][~want], w[0][~want])      # no renormalisation
    assert np.all(w2[0][want] == 0.0)


def test_monotone_in_n_and_per_call():
    rng = np.random.default_rng(7)
    T, K, E = 6, 8, 40
    ids = np.stack([np.sort(rng.choice(E, K, replace=False)) for _ in range(T)])
    w = rng.random((T, K)).astype(np.float32)
    prev = None
    for n in range(1, K):
        _, sk = oracle.tail_skip(ids, w, n)
        if prev is not None:
            assert not (sk & ~prev).any()          # a larger n never skips more
        prev = sk
        # per call: an expert is skipped in every token that picked it, or in none
        for e in np.unique(ids):
            marks = sk[ids == e]
            assert marks.all() or not marks.any()


def test_invariant_to_the_order_of_picks():
    rng = np.random.default_rng(3)
    T, K = 4, 8
    ids = np.stack([np.sort(rng.choice(100, K, replace=False)) for _ in range(T)])
    w = rng.random((T, K)).astype(np.float32)
    _, sk = oracle.tail_skip(ids, w, 5)
    perm = rng.permutation(K)
    _, sk2 = oracle.tail_skip(ids[:, perm], w[:, perm], 5)
    assert np.array_equal(sk[:, perm], sk2)


def test_forward_drops_exactly_the_skipped_terms():
    """out(tail-skip) + sum over skipped picks of w y = out(all picks), the
    layer being linear in the routed terms for fixed routing."""
    dims = gen.TOY
    planes = gen.draw_layer(dims, 2)
    xb = gen.draw_tokens(dims, 3, 2, "bf16")
    full = oracle.moe_forward(dims, planes, xb, want_y=True)
    w2, sk = oracle.tail_skip(full["ids"], full["w"], 2)
    assert sk.any() and not sk.all()
    part = oracle.moe_forward(dims, planes, xb, ids=full["ids"], w=w2)
    dropped = np.einsum("tk,tkh->th", np.where(sk, full["w"], 0.0), full["y"].astype(np.float64))
    np.testing.assert_allclose(part["out"] + dropped, full["out"], rtol=1e-5, atol=1e-6)

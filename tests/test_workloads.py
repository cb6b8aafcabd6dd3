"""The seeded generator: shapes, formats, and the workload properties
(cosine-0.9 pairs, Zipf skew) the synthetic inputs are meant to have."""
import numpy as np

import oracle
from workloads import gen


def test_layer_planes_shapes_and_formats():
    d = gen.TOY
    L = gen.draw_layer(d, 0)
    H, E, I, Is = d.hidden, d.n_experts, d.inter, d.shared_inter
    assert L["router"].shape == (E + 1, H) and L["router"].dtype == np.uint16
    assert L["gu_q"].shape == (E, 2 * I, H // 2) and L["gu_q"].dtype == np.uint8
    assert L["gu_s"].shape == (E, 2 * I, H // 32) and L["gu_s"].dtype == np.uint16
    assert L["dn_q"].shape == (E, H, I // 2)
    assert L["dn_s"].shape == (E, H, I // 32)
    assert L["sh_gu_q"].shape == (2 * Is, H // 2)
    assert L["sh_dn_s"].shape == (H, Is // 32)
    assert L["router_bias"] is None
    s = L["gu_s"].view(np.float16).astype(np.float64)
    assert np.all(s >= 0) and abs(np.sqrt((s * s).mean()) - 0.02) < 0.002


def test_draws_are_seeded_and_distinct():
    d = gen.TOY
    a, b, c = gen.draw_layer(d, 3), gen.draw_layer(d, 3), gen.draw_layer(d, 4)
    assert np.array_equal(a["gu_q"], b["gu_q"]) and not np.array_equal(a["gu_q"], c["gu_q"])


def test_nibbles_uniform_on_int4_range():
    L = gen.draw_layer(gen.TOY, 0)
    q = L["gu_q"].ravel()
    nib = np.concatenate([q & 15, q >> 4])
    counts = np.bincount(nib, minlength=16) / nib.size
    assert np.all(np.abs(counts - 1 / 16) < 0.005)


def test_pairs_have_cosine_point_nine():
    r = gen.draw_tokens(gen.QWEN, 16, 0, "pairs")
    for p in range(8):
        a, b = r[2 * p].astype(np.float64), r[2 * p + 1].astype(np.float64)
        cos = a @ b / np.linalg.norm(a) / np.linalg.norm(b)
        assert abs(cos - 0.9) < 1e-5
        assert abs(np.sqrt((a * a).mean()) - 1.0) < 1e-5


def test_zipf_bias_form():
    b = gen.zipf_bias(256, 0.5, 0)
    ranks = np.rint(np.exp(-b / (0.5 * gen.ZIPF_S))).astype(int)
    assert sorted(ranks) == list(range(1, 257))


def test_decode16_skew_about_80_20():
    d = gen.QWEN
    L = gen.draw_layer(d, 0, bias="zipf", alpha=gen.ALPHA_DECODE16)
    x = oracle.rmsnorm(gen.draw_tokens(d, 2048, 123, "resid"))
    logits, _ = oracle.router(x, L["router"], L["router_bias"])
    ids, _, _ = oracle.select(logits, d.top_k)
    c = np.sort(np.bincount(ids.ravel(), minlength=d.n_experts))[::-1]
    share = c[:51].sum() / c.sum()
    assert 0.78 <= share <= 0.82, share


def test_prefill_loads_up_to_about_300():
    cfg = gen.CONFIGS["prefill"]
    d = cfg.dims
    L = gen.draw_layer(d, 0, bias="zipf", alpha=cfg.alpha)
    x = oracle.rmsnorm(gen.draw_tokens(d, cfg.tokens, 0, "resid"))
    logits, _ = oracle.router(x, L["router"], L["router_bias"])
    ids, _, _ = oracle.select(logits, d.top_k)
    loads = np.bincount(ids.ravel(), minlength=d.n_experts)
    assert 270 <= loads.max() <= 330 and loads.min() >= 5, (loads.min(), loads.max())

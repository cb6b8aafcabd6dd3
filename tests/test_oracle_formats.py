"""Pins of the oracle's number formats and int4 dequantisation."""
import os

import numpy as np
import pytest
import torch

import oracle
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_f16_decode_all_bit_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_decode_against_torch():
    rng = np.random.default_rng(1)
    bits = np.concatenate([rng.integers(0, 65536, 4000).astype(np.uint16),
                           np.array([0x0000, 0x8000, 0x0001, 0x3F80, 0xC000, 0x7F80, 0xFF80],
                                    dtype=np.uint16)])
    got = oracle.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_rounding_hand_cases():
    cases = {
        1.0: 0x3F80,
        1.00390625: 0x3F80,        # 1 + 2^-8: exactly half an ulp, ties to even (down)
        1.01171875: 0x3F82,        # 1 + 3*2^-8: half an ulp above 0x3F81, ties to even (up)
        1.005859375: 0x3F81,       # 1 + 1.5*2^-8: above the half, rounds up
        -2.0: 0xC000,
        3.0e38: 0x7F62,            # 3e38 = 0x7F61B1E6 -> rounds up to 0x7F62
        float("inf"): 0x7F80,
    }
    for v, want in cases.items():
        got = int(oracle.round_bf16(np.array([v], dtype=np.float32))[0])
        assert got == want, (v, hex(got), hex(want))


def test_bf16_rounding_against_torch():
    rng = np.random.default_rng(2)
    a = np.concatenate([rng.normal(0, 1, 20000), rng.normal(0, 1e-38, 1000),
                        rng.normal(0, 1e30, 1000)]).astype(np.float32)
    got = oracle.round_bf16(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "dequant_bytes.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            b, s, e0, e1 = line.split()
            rows.append((int(b, 16), int(s, 16), float(e0), float(e1)))
    return rows


def test_dequant_hand_computed_bytes():
    rows = _golden_rows()
    assert len(rows) >= 10
    for b, s, e0, e1 in rows:
        q = np.zeros((16,), dtype=np.uint8)
        q[0] = b
        sc = np.array([s], dtype=np.uint16)
        W = oracle.dequant_matrix(q, sc, 1, 32)
        assert W[0, 0] == np.float32(e0), (hex(b), hex(s), W[0, 0], e0)
        assert W[0, 1] == np.float32(e1), (hex(b), hex(s), W[0, 1], e1)


def test_nibble_matches_xor_rule_for_every_byte():
    q = np.arange(256, dtype=np.uint8)
    for j in range(512):
        raw = (int(q[j // 2]) >> (4 * (j & 1))) & 0xF
        x = raw ^ 0x8
        signed = x - 16 if x >= 8 else x
        assert oracle.nibble(q, j) == signed


def test_dequant_scale_group_boundaries():
    # a row of 96 elements: three scale groups; element j in group j // 32
    rows, cols = 2, 96
    q = np.full((rows, cols // 2), 0xF9, dtype=np.uint8)   # even elements 1, odd 7
    s = np.array([[0x3C00, 0x4000, 0x3800], [0x4400, 0x0000, 0xBC00]], dtype=np.uint16)
    W = oracle.dequant_matrix(q, s, rows, cols)
    scale = np.array([[1.0, 2.0, 0.5], [4.0, 0.0, -1.0]], dtype=np.float32)
    for r in range(rows):
        for j in range(cols):
            want = scale[r, j // 32] * (1.0 if j % 2 == 0 else 7.0)
            assert W[r, j] == np.float32(want)


def test_dequant_matches_brute_random():
    rng = np.random.default_rng(3)
    rows, cols = 8, 256
    q = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    s = np.abs(rng.normal(0, 0.02, (rows, cols // 32))).astype(np.float16).view(np.uint16)
    W = oracle.dequant_matrix(q, s, rows, cols)
    ref = brute.dequant_xor(q, s, rows, cols)
    assert np.array_equal(W.astype(np.float64), ref)       # exact in fp32

"""Seeded draws of MoE layers and tokens in their storage formats.

Storage formats (the packed-weight layout both the CUDA library and the CPU
oracle read; the library's header states it in full):

* router      uint16 [E+1][H]   bf16 bit patterns; row E is the shared-expert
                                gate vector (the router and the shared gate
                                form one product, Strata "Qwen3.6-35B-A3B:
                                pictures, several requests at once and speed",
                                section "Speed").
* router_bias float32 [E]       or None.
* gu_q        uint8 [E][2I][H/2]  int4 offset-binary nibbles, two per byte,
                                  rows interleaved gate/up (row 2i = gate i,
                                  row 2i+1 = up i).
* gu_s        uint16 [E][2I][H/32] fp16 scale bit patterns, one per 32
                                  consecutive input elements of a row.
* dn_q        uint8 [E][H][I/2],  dn_s uint16 [E][H][I/32]
* sh_*        the same four planes for the shared expert (one expert, Is).

Because a uniformly random byte has two independent, uniformly random nibbles,
drawing the packed planes as uniform bytes gives weights uniform on the
integers [-8, 7] without any packing arithmetic here.  Scales are |N(0, 0.02)|
rounded to fp16 by numpy's round-to-nearest-even cast.

Nothing in this module routes, dequantises, normalises or multiplies: the
residual-stream activations of the Qwen-shaped workloads are drawn as fp32
N(0, 1) and the path under test (or the oracle) applies the RMSNorm itself.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

ZIPF_S = 1.1

# Strength of the Zipf(s=1.1) logit bias b_e = -alpha * s * ln(rank_e).  The two
# values were chosen with tests/golden/calibrate_zipf.py, which routes synthetic
# tokens through the oracle:
#   ALPHA_DECODE16 = 0.505 puts 80% of the selections on the 20% most selected
#     experts (over 4,096 tokens);
#   ALPHA_PREFILL = 0.165 gives a largest expert load of about 300 rows at
#     T=2048 (299 for seed 0; the smallest load is then 26).  A log-rank bias
#     cannot also bring the smallest load down to about 10 without pushing the
#     largest past 500, so the largest load, which sets the tile work, is the
#     one matched.
# tests/test_workloads.py re-checks both properties.
ALPHA_DECODE16 = 0.505
ALPHA_PREFILL = 0.165

_TAG_LAYER, _TAG_TOKENS, _TAG_BIAS, _TAG_IDS = 1, 2, 3, 4


@dataclass(frozen=True)
class LayerDims:
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    shared_inter: int
    group: int = 32


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    dims: LayerDims
    tokens: int
    token_kind: str          # "bf16" (x drawn directly) | "resid" | "pairs"
    bias: str                # "none" | "zipf"
    alpha: float = 0.0
    seeds: tuple = (0,)
    description: str = ""
    extra: dict = field(default_factory=dict)


QWEN = LayerDims(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512)
TOY = LayerDims(hidden=512, n_experts=32, top_k=4, inter=128, shared_inter=128)

CONFIGS = {
    "toy": WorkloadConfig(
        "toy", TOY, 4, "bf16", "none", seeds=(0,),
        description="toy MoE layer: T=4, H=512, 32 experts, top-4, I=Is=128"),
    "decode1": WorkloadConfig(
        "decode1", QWEN, 1, "resid", "none", seeds=tuple(range(10)),
        description="Qwen3.6-35B-A3B-shaped MoE layer, decode T=1, "
                    "10 distinct layers (seeds 0..9), uniform routing"),
    "decode16": WorkloadConfig(
        "decode16", QWEN, 16, "pairs", "zipf", alpha=ALPHA_DECODE16, seeds=(0,),
        description="decode T=16: 8 requests x 2 MTP tokens, cosine-0.9 pairs, "
                    "Zipf(1.1) router bias"),
    "stack": WorkloadConfig(
        "stack", QWEN, 1, "resid", "none", seeds=tuple(range(40)),
        description="40-layer MoE stack, residual + RMSNorm between layers, T=1 or 4"),
    "prefill": WorkloadConfig(
        "prefill", QWEN, 2048, "resid", "zipf", alpha=ALPHA_PREFILL, seeds=(0,),
        description="prefill T=2048, Zipf(1.1)-skewed routing"),
}


def _rng(seed: int, tag: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), tag])))


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 draws to bf16 (torch's round-to-nearest-even cast) and
    return the bit patterns as uint16."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _fp16_abs_normal(rng, shape, std):
    return np.abs(rng.normal(0.0, std, size=shape)).astype(np.float16).view(np.uint16)


def zipf_bias(n_experts: int, alpha: float, seed: int) -> np.ndarray:
    """Router logit bias -alpha * s * ln(rank) over a seeded random order of
    the experts (rank 1 is the most favoured expert)."""
    rng = _rng(seed, _TAG_BIAS)
    rank = rng.permutation(n_experts).astype(np.float64) + 1.0
    return (-alpha * ZIPF_S * np.log(rank)).astype(np.float32)


def draw_layer(dims: LayerDims, seed: int, bias: str = "none", alpha: float = 0.0,
               router_std: float = 0.02, scale_std: float = 0.02) -> dict:
    """One MoE layer's weights in storage format (see the module docstring)."""
    H, E, I, Is, G = dims.hidden, dims.n_experts, dims.inter, dims.shared_inter, dims.group
    rng = _rng(seed, _TAG_LAYER)
    layer = {
        "router": _bf16_bits(rng.normal(0.0, router_std, size=(E + 1, H)).astype(np.float32)),
        "gu_q": rng.integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8),
        "gu_s": _fp16_abs_normal(rng, (E, 2 * I, H // G), scale_std),
        "dn_q": rng.integers(0, 256, size=(E, H, I // 2), dtype=np.uint8),
        "dn_s": _fp16_abs_normal(rng, (E, H, I // G), scale_std),
        "sh_gu_q": rng.integers(0, 256, size=(2 * Is, H // 2), dtype=np.uint8),
        "sh_gu_s": _fp16_abs_normal(rng, (2 * Is, H // G), scale_std),
        "sh_dn_q": rng.integers(0, 256, size=(H, Is // 2), dtype=np.uint8),
        "sh_dn_s": _fp16_abs_normal(rng, (H, Is // G), scale_std),
        "router_bias": zipf_bias(E, alpha, seed) if bias == "zipf" else None,
    }
    return layer


def draw_tokens(dims: LayerDims, T: int, seed: int, kind: str) -> np.ndarray:
    """Activations for T tokens.

    kind "bf16":  x, bf16 bit patterns of N(0,1) draws, uint16 [T][H]
    kind "resid": r, fp32 N(0,1) [T][H]; the path RMS-normalises it
    kind "pairs": r, fp32 [T][H], T even: tokens 2p and 2p+1 have cosine
                  exactly 0.9 (an MTP draft following its request's token):
                  with a, z unit vectors, z orthogonal to a,
                  r_2p = sqrt(H) a and r_2p+1 = sqrt(H) (0.9 a + sqrt(0.19) z)
    """
    H = dims.hidden
    rng = _rng(seed, _TAG_TOKENS)
    if kind == "bf16":
        return _bf16_bits(rng.normal(0.0, 1.0, size=(T, H)).astype(np.float32))
    if kind == "resid":
        return rng.normal(0.0, 1.0, size=(T, H)).astype(np.float32)
    if kind == "pairs":
        assert T % 2 == 0
        out = np.empty((T, H), dtype=np.float64)
        for p in range(T // 2):
            a = rng.normal(size=H)
            z = rng.normal(size=H)
            a /= np.linalg.norm(a)
            z -= a * np.dot(a, z)
            z /= np.linalg.norm(z)
            out[2 * p] = np.sqrt(H) * a
            out[2 * p + 1] = np.sqrt(H) * (0.9 * a + np.sqrt(1.0 - 0.81) * z)
        return out.astype(np.float32)
    raise ValueError(kind)


def draw_ids(T: int, n_experts: int, top_k: int, seed: int):
    """Forced routing: per token top_k distinct expert ids in ascending order
    and positive weights (any values; the layer does not require them to sum
    to one when they are forced)."""
    rng = _rng(seed, _TAG_IDS)
    ids = np.empty((T, top_k), dtype=np.int32)
    for t in range(T):
        ids[t] = np.sort(rng.choice(n_experts, size=top_k, replace=False))
    w = rng.uniform(0.05, 1.0, size=(T, top_k)).astype(np.float32)
    return ids, w


def workload(name: str) -> WorkloadConfig:
    return CONFIGS[name]

"""Emulation of an 8-bit-activation prefill path (test infrastructure only,
for the tolerance study such a path needs before it is built).

The pages' own version (Strata, "Strata on an Intel Arc", section "Arc Pro
B70: the fused int8 expert path for the prompt") quantizes the activations
in blocks of 32 and decodes the quantized weights straight into the 8-bit
matrix operand.  On this GPU the 8-bit tensor path with block scales is
MXFP8: e4m3 elements with one power-of-two (UE8M0) scale per 32 along K for
each operand.  The emulated scheme:

  activations  per token and 32-block: scale 2^(floor(log2 amax) - 8),
               elements e4m3(x / scale)
  weights      s = fp16 group scale = 2^e * m with m in [1, 2): block scale
               2^e, elements e4m3((q - 8) * m)  (q - 8 is exact in e4m3;
               the product with m is the one rounding)
  products     fp32 sums of (a_elem * a_scale) * (w_elem * w_scale)

everything else as the exact layer (router, top-K, SwiGLU, shared gate,
combine in the oracle's order).  Written from the OCP 8-bit floating-point
and microscaling definitions: e4m3 has a 4-bit exponent of bias 7, a 3-bit
mantissa, normals from 2^-6 to 448, subnormals in steps of 2^-9, and no
infinity; conversion rounds to nearest, ties to even, and saturates to
+-448.  Plain numpy in float64; nothing here is used by the CUDA library.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6
E4M3_MANT_BITS = 3


def e4m3_round(v):
    """Nearest e4m3 value (ties to even), saturated to +-448; NaN stays NaN."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    out = np.zeros_like(a)
    nz = a > 0
    # exponent of the value's binade, clamped below to the subnormal range
    e = np.floor(np.log2(np.where(nz, a, 1.0)))
    e = np.maximum(e, E4M3_MIN_NORMAL_EXP)
    step = np.exp2(e - E4M3_MANT_BITS)             # spacing of e4m3 values there
    r = np.round(a / step) * step                  # numpy rounds half to even
    out = np.where(nz, r, 0.0)
    out = np.minimum(out, E4M3_MAX)
    out = np.where(np.isnan(a), np.nan, out)
    return np.copysign(out, v)


def e4m3_values():
    """Every finite e4m3 value, from the bit fields (sign, exponent, mantissa)."""
    vals = []
    for s in (1.0, -1.0):
        for ex in range(16):
            for m in range(8):
                if ex == 15 and m == 7:
                    continue                        # the NaN code
                if ex == 0:
                    v = m / 8.0 * 2.0 ** (1 - 7)    # subnormal
                else:
                    v = (1.0 + m / 8.0) * 2.0 ** (ex - 7)
                vals.append(s * v)
    return np.array(sorted(set(vals)))


def mx_quantize(x, block: int = 32):
    """MXFP8 of rows of x along the last axis: (elements, scales), with
    x ~= elements * repeat(scales, block).  A block of zeros gets scale 1."""
    x = np.asarray(x, dtype=np.float64)
    *lead, n = x.shape
    assert n % block == 0
    xb = x.reshape(*lead, n // block, block)
    amax = np.max(np.abs(xb), axis=-1, keepdims=True)
    ex = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, 0.0)
    scale = np.exp2(ex)
    el = e4m3_round(xb / scale)
    return el.reshape(*lead, n), scale[..., 0]


def weight_mx(q, s_f16_bits, block: int = 32):
    """Weights of one matrix: q int8 [rows][cols] (values -8..7), fp16 scale
    bits [rows][cols/32] -> effective float64 weights of the MXFP8 scheme."""
    s = np.asarray(s_f16_bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    ex = np.floor(np.log2(np.where(s > 0, s, 1.0)))
    bscale = np.exp2(ex)                            # power-of-two part: block scale
    m = np.where(s > 0, s / bscale, 0.0)            # mantissa part, in [1, 2)
    qq = np.asarray(q, dtype=np.float64)
    rows, cols = qq.shape
    mm = np.repeat(m, block, axis=1)
    el = e4m3_round(qq * mm)
    return el * np.repeat(bscale, block, axis=1)


def act_mx(x, block: int = 32):
    """Effective float64 activations of the MXFP8 scheme."""
    el, sc = mx_quantize(x, block)
    return el * np.repeat(sc, block, axis=-1)


# ------------------------------------------------------------------ layer
def unpack_q(packed):
    """Signed int4 values (u - 8) of packed rows: byte b holds element 2b in
    bits 0-3 and element 2b + 1 in bits 4-7, offset-binary u = q + 8."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = (p & 0x0F).astype(np.int8) - 8
    hi = (p >> 4).astype(np.int8) - 8
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def _weights(q_packed, s_bits, quantize):
    q = unpack_q(q_packed).astype(np.float64)
    if quantize:
        return weight_mx(q, s_bits)
    s = np.asarray(s_bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    return q * np.repeat(s, 32, axis=1)


def _bf16(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def _ffn(x, Wgu, Wd, quantize):
    """SwiGLU expert in float64 on activations x [n][H]; gate/up rows are
    interleaved (row 2i gate i, row 2i + 1 up i)."""
    xa = act_mx(x) if quantize else x
    gu = xa @ Wgu.T
    g, u = gu[:, 0::2], gu[:, 1::2]
    h = g / (1.0 + np.exp(-g)) * u
    ha = act_mx(h) if quantize else h
    return ha @ Wd.T


def layer_forward(dims, planes, xb, ids, w, sig, quantize: bool = True):
    """out [T][H] (float64) of the layer with the given routing (ids, w,
    sigmoid gates sig), the experts' products in the MXFP8 scheme when
    quantize, else exact; the combine sums the picks in ascending k."""
    x = _bf16(xb)
    T, H = x.shape
    K = ids.shape[1]
    y = np.zeros((T, K, H))
    for e in np.unique(ids):
        tk = np.argwhere(ids == e)
        Wgu = _weights(planes["gu_q"][e], planes["gu_s"][e], quantize)
        Wd = _weights(planes["dn_q"][e], planes["dn_s"][e], quantize)
        y[tk[:, 0], tk[:, 1]] = _ffn(x[tk[:, 0]], Wgu, Wd, quantize)
    S = _ffn(x, _weights(planes["sh_gu_q"], planes["sh_gu_s"], quantize),
             _weights(planes["sh_dn_q"], planes["sh_dn_s"], quantize), quantize)
    out = np.zeros((T, H))
    for k in range(K):
        out += np.asarray(w, dtype=np.float64)[:, k:k + 1] * y[:, k]
    return out + np.asarray(sig, dtype=np.float64)[:, None] * S

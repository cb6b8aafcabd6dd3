"""float64 numpy brute force of the MoE layer, used only to pin the oracle.

It shares the oracle's reading of the method (routing by the K largest
logits with ties to the lower id, renormalised softmax, SwiGLU, sigmoid gate)
but none of its arithmetic: everything here is float64 library matmuls on
dequantised matrices, so its result is the exact value up to ~1e-15 and the
oracle's fp32 result must sit within fp32 rounding of it.
"""
import numpy as np
import torch


def bf16_bits_to_f64(bits):
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).to(torch.float64).numpy()


def f16_bits_to_f64(bits):
    return np.ascontiguousarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def dequant_xor(q, s, rows, cols):
    """Dequantise with the page's XOR rule: a raw nibble XOR 8, read as a
    4-bit two's-complement integer, is the signed weight."""
    q = np.asarray(q, dtype=np.uint8).reshape(rows, cols // 2)
    lo = (q & 0x0F) ^ 0x08
    hi = (q >> 4) ^ 0x08
    nib = np.empty((rows, cols), dtype=np.int64)
    nib[:, 0::2] = lo
    nib[:, 1::2] = hi
    signed = np.where(nib >= 8, nib - 16, nib)
    scale = f16_bits_to_f64(np.asarray(s).reshape(rows, cols // 32))
    return signed.astype(np.float64) * np.repeat(scale, 32, axis=1)


def silu(g):
    return g / (1.0 + np.exp(-g))


def expert(x, Wgu, Wd):
    gu = Wgu @ x
    h = silu(gu[0::2]) * gu[1::2]
    return h, Wd @ h


def layer(dims, L, x_bits, ids=None, w=None):
    """Returns out [T][H] float64 plus the routing it used and the gap
    between the K-th and (K+1)-th logits."""
    H, E, K, I, Is = dims.hidden, dims.n_experts, dims.top_k, dims.inter, dims.shared_inter
    x = bf16_bits_to_f64(x_bits)
    T = x.shape[0]
    R = bf16_bits_to_f64(L["router"])
    logits = x @ R[:E].T
    if L.get("router_bias") is not None:
        logits = logits + np.asarray(L["router_bias"], dtype=np.float64)
    s = x @ R[E]
    gap = np.full((T,), np.inf)
    if ids is None:
        ids = np.empty((T, K), dtype=np.int64)
        w = np.empty((T, K))
        for t in range(T):
            order = sorted(range(E), key=lambda e: (-logits[t, e], e))
            sel = sorted(order[:K])
            if K < E:
                gap[t] = logits[t, order[K - 1]] - logits[t, order[K]]
            m = max(logits[t, e] for e in sel)
            ex = np.array([np.exp(logits[t, e] - m) for e in sel])
            ids[t] = sel
            w[t] = ex / ex.sum()
    sig = 1.0 / (1.0 + np.exp(-s))
    Wsgu = dequant_xor(L["sh_gu_q"], L["sh_gu_s"], 2 * Is, H)
    Wsd = dequant_xor(L["sh_dn_q"], L["sh_dn_s"], H, Is)
    out = np.zeros((T, H))
    cache = {}
    for t in range(T):
        for k in range(K):
            e = int(ids[t, k])
            if e not in cache:
                cache[e] = (dequant_xor(L["gu_q"][e], L["gu_s"][e], 2 * I, H),
                            dequant_xor(L["dn_q"][e], L["dn_s"][e], H, I))
            _, y = expert(x[t], *cache[e])
            out[t] += w[t, k] * y
        _, S = expert(x[t], Wsgu, Wsd)
        out[t] += sig[t] * S
    return {"out": out, "ids": np.asarray(ids), "w": np.asarray(w), "gap": gap, "sig": sig,
            "logits": logits}

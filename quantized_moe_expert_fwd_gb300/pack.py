"""Host-side packing of canonical MoE weights into the library's layout.

Canonical form (what a model file gives after its own decoding):
  router      [H][E] values (fp32 or bf16 bit patterns) and the shared-expert
              gate vector [H]
  an expert   gate q [I][H], up q [I][H], down q [H][I] as signed int4 values in
              [-8, 7] (int8 arrays) with fp16 scales [rows][cols/32]
Packed form (include/strata_moe.h): router [E+1][H] (row E = gate vector);
gate/up rows interleaved (row 2i gate, 2i+1 up); nibbles offset-binary, the
even element of a pair in the low nibble.  Runs once per model load, on the
host, outside any timed path.
"""
from __future__ import annotations

import numpy as np
import torch


def pack_int4(q) -> np.ndarray:
    """int8 [rows][cols] with values in [-8, 7] -> uint8 [rows][cols/2]."""
    q = np.asarray(q)
    if q.ndim < 1 or q.shape[-1] % 2:
        raise ValueError("the last axis must have even length")
    if q.min(initial=0) < -8 or q.max(initial=0) > 7:
        raise ValueError("int4 values must lie in [-8, 7]")
    u = (q.astype(np.int16) + 8).astype(np.uint8)
    return (u[..., 0::2] | (u[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(packed) -> np.ndarray:
    """Inverse of pack_int4."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = (p & 0x0F).astype(np.int8) - 8
    out[..., 1::2] = (p >> 4).astype(np.int8) - 8
    return out


def _f16_bits(s) -> np.ndarray:
    s = np.asarray(s)
    if s.dtype == np.uint16:
        return s
    return s.astype(np.float16).view(np.uint16)


def _bf16_bits(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return a
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def pack_gate_up(q_gate, s_gate, q_up, s_up):
    """Interleave gate and up rows: packed row 2i = gate i, 2i+1 = up i."""
    qg, qu = np.asarray(q_gate), np.asarray(q_up)
    if qg.shape != qu.shape:
        raise ValueError("gate and up must have the same shape")
    rows = qg.shape[-2]
    q = np.empty(qg.shape[:-2] + (2 * rows, qg.shape[-1]), dtype=np.int8)
    q[..., 0::2, :] = qg
    q[..., 1::2, :] = qu
    sg, su = _f16_bits(s_gate), _f16_bits(s_up)
    s = np.empty(sg.shape[:-2] + (2 * rows, sg.shape[-1]), dtype=np.uint16)
    s[..., 0::2, :] = sg
    s[..., 1::2, :] = su
    return pack_int4(q), s


def pack_router(router_he, gate_h):
    """[H][E] router and [H] shared gate -> bf16 [E+1][H]."""
    r = _bf16_bits(router_he)
    g = _bf16_bits(gate_h).reshape(1, -1)
    return np.ascontiguousarray(np.concatenate([r.T, g], axis=0))


def pack_layer(canon: dict) -> dict:
    """canon keys: router [H][E], gate_vec [H], router_bias [E] or None,
    q_gate/s_gate, q_up/s_up [E][I][H] (+ scales [E][I][H/32]), q_down/s_down
    [E][H][I], and sh_q_gate, sh_s_gate, sh_q_up, sh_s_up, sh_q_down,
    sh_s_down for the shared expert."""
    gu_q, gu_s = pack_gate_up(canon["q_gate"], canon["s_gate"], canon["q_up"], canon["s_up"])
    sh_gu_q, sh_gu_s = pack_gate_up(canon["sh_q_gate"], canon["sh_s_gate"], canon["sh_q_up"],
                                    canon["sh_s_up"])
    bias = canon.get("router_bias")
    return {
        "router": pack_router(canon["router"], canon["gate_vec"]),
        "router_bias": None if bias is None else np.asarray(bias, dtype=np.float32),
        "gu_q": gu_q, "gu_s": gu_s,
        "dn_q": pack_int4(canon["q_down"]), "dn_s": _f16_bits(canon["s_down"]),
        "sh_gu_q": sh_gu_q, "sh_gu_s": sh_gu_s,
        "sh_dn_q": pack_int4(canon["sh_q_down"]), "sh_dn_s": _f16_bits(canon["sh_s_down"]),
    }


def quantize_symmetric(w, group: int = 32):
    """Float weights [rows][cols] -> (int8 q in [-8, 7], fp16 scales
    [rows][cols/group]): per group s = max|w| / 8 rounded to fp16 and
    q = clip(round(w / s), -8, 7).  A convenience for real weights; the
    synthetic workloads draw q and s directly."""
    w = np.asarray(w, dtype=np.float32)
    rows, cols = w.shape
    g = w.reshape(rows, cols // group, group)
    s = (np.abs(g).max(axis=2) / 8.0).astype(np.float16)
    sf = s.astype(np.float32)
    safe = np.where(sf == 0, 1.0, sf)
    q = np.clip(np.rint(g / safe[:, :, None]), -8, 7).astype(np.int8).reshape(rows, cols)
    return q, s.view(np.uint16)

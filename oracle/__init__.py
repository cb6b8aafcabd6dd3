"""CPU oracle of the routed MoE FFN forward (test infrastructure only).

A plain fp32 C implementation (moe_oracle.c) behind numpy wrappers.  Only the
tests, the smoke check and the bench's CPU-baseline leg use it; the CUDA
library never imports, links or reads it, and it never reads anything the
CUDA library produced.  See moe_oracle.c for the arithmetic rules and the
passages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over independent experts/tokens;
    -ffp-contract=off keeps every multiply and add separately rounded)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OrcLayer(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "router", "router_bias", "gu_q", "gu_s", "dn_q", "dn_s",
        "sh_gu_q", "sh_gu_s", "sh_dn_q", "sh_dn_s")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            _lib.orc_bf16_to_f32.restype = ctypes.c_float
            _lib.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            _lib.orc_f16_to_f32.restype = ctypes.c_float
            _lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            _lib.orc_f32_to_bf16.restype = ctypes.c_uint16
            _lib.orc_f32_to_bf16.argtypes = [ctypes.c_float]
            _lib.orc_round_bf16.argtypes = [ctypes.c_int64, P, P]
            _lib.orc_nibble.restype = I
            _lib.orc_nibble.argtypes = [P, I]
            _lib.orc_dequant_row.argtypes = [P, P, I, P]
            _lib.orc_dequant_matrix.argtypes = [P, P, I, I, P]
            _lib.orc_rmsnorm.argtypes = [I, I, P, ctypes.c_float, P]
            _lib.orc_router.argtypes = [I, I, I, P, P, P, P, P]
            _lib.orc_select.argtypes = [I, I, I, P, P, P, P]
            _lib.orc_sigmoid.restype = ctypes.c_float
            _lib.orc_sigmoid.argtypes = [ctypes.c_float]
            _lib.orc_swiglu.restype = ctypes.c_float
            _lib.orc_swiglu.argtypes = [ctypes.c_float, ctypes.c_float]
            _lib.orc_permute.argtypes = [I, I, I, P, P, P, P, P]
            _lib.orc_expert_dense.argtypes = [I, I, P, P, P, P, P, P]
            _lib.orc_moe_forward.restype = I
            _lib.orc_moe_forward.argtypes = [I, I, I, I, I, ctypes.POINTER(OrcLayer), I,
                                             P, I, P, P, P, P, P, P, P, P, P, I]
        return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ formats
def bf16_to_f32(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    f = lib().orc_bf16_to_f32
    return np.array([f(int(b)) for b in bits.ravel()], dtype=np.float32).reshape(bits.shape)


def bf16_array_to_f32(bits) -> np.ndarray:
    """Vectorised decode for large arrays (the same bit rule: bits << 16)."""
    bits = _c(bits, np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def f16_to_f32(bits) -> np.ndarray:
    bits = _c(bits, np.uint16)
    f = lib().orc_f16_to_f32
    return np.array([f(int(b)) for b in bits.ravel()], dtype=np.float32).reshape(bits.shape)


def round_bf16(a) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    lib().orc_round_bf16(a.size, _p(a), _p(out))
    return out


def nibble(q, j: int) -> int:
    q = _c(q, np.uint8)
    return lib().orc_nibble(_p(q), j)


def dequant_matrix(q, s, rows: int, cols: int) -> np.ndarray:
    q = _c(q, np.uint8)
    s = _c(s, np.uint16)
    out = np.empty((rows, cols), dtype=np.float32)
    lib().orc_dequant_matrix(_p(q), _p(s), rows, cols, _p(out))
    return out


# ------------------------------------------------------------------- layer
def rmsnorm(r, eps: float = 1e-6) -> np.ndarray:
    r = _c(r, np.float32)
    T, H = r.shape
    x = np.empty((T, H), dtype=np.uint16)
    lib().orc_rmsnorm(T, H, _p(r), ctypes.c_float(eps), _p(x))
    return x


def router(x, router_bits, bias=None):
    x = _c(x, np.uint16)
    rb = _c(router_bits, np.uint16)
    T, H = x.shape
    E = rb.shape[0] - 1
    b = None if bias is None else _c(bias, np.float32)
    logits = np.empty((T, E), dtype=np.float32)
    gate = np.empty((T,), dtype=np.float32)
    lib().orc_router(T, H, E, _p(x), _p(rb), _p(b), _p(logits), _p(gate))
    return logits, gate


def select(logits, K: int):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    ids = np.empty((T, K), dtype=np.int32)
    w = np.empty((T, K), dtype=np.float32)
    gap = np.empty((T,), dtype=np.float32)
    lib().orc_select(T, E, K, _p(logits), _p(ids), _p(w), _p(gap))
    return ids, w, gap


def tail_skip(ids, w, n: int):
    """Tail-skip of one call's routing (PolyStrata, "Models and backends",
    section "What was tuned": an expert that every token of a call ranks at
    place n + 1 or later of its picks is left out, and the picks that stay
    keep the weights the router gave them; prompt batches are not touched).

    ids, w: [T][K] routing of the call.  A pick's place is 1 + the number of
    its token's picks with a larger weight, or an equal weight and a lower
    id (the selection's own order: larger logit first, ties to the lower
    id).  Returns (w2, skipped): w with the left-out picks' weights set to
    0, and a [T][K] bool mask of those picks.  n <= 0 or n >= K leaves every
    pick (n = 0 is "off").  Plain loops: calls have at most a few hundred
    picks."""
    ids = np.asarray(ids, dtype=np.int64)
    w = np.asarray(w, dtype=np.float32)
    T, K = ids.shape
    skipped = np.zeros((T, K), dtype=bool)
    if n <= 0 or n >= K:
        return w.copy(), skipped
    place = np.zeros((T, K), dtype=np.int64)
    for t in range(T):
        for k in range(K):
            before = 0
            for j in range(K):
                if w[t, j] > w[t, k] or (w[t, j] == w[t, k] and ids[t, j] < ids[t, k]):
                    before += 1
            place[t, k] = before + 1
    kept = set()
    for t in range(T):
        for k in range(K):
            if place[t, k] <= n:
                kept.add(int(ids[t, k]))
    for t in range(T):
        for k in range(K):
            skipped[t, k] = int(ids[t, k]) not in kept
    w2 = w.copy()
    w2[skipped] = 0.0
    return w2, skipped


def sigmoid(s: float) -> float:
    return float(lib().orc_sigmoid(ctypes.c_float(s)))


def swiglu(g: float, u: float) -> float:
    return float(lib().orc_swiglu(ctypes.c_float(g), ctypes.c_float(u)))


def permute(ids, E: int):
    ids = _c(ids, np.int32)
    T, K = ids.shape
    counts = np.empty((E,), dtype=np.int32)
    offsets = np.empty((E + 1,), dtype=np.int32)
    perm = np.empty((T * K,), dtype=np.int32)
    inv = np.empty((T * K,), dtype=np.int32)
    lib().orc_permute(T, K, E, _p(ids), _p(counts), _p(offsets), _p(perm), _p(inv))
    return counts, offsets, perm, inv


def expert_dense(x_f32, Wgu, Wd):
    x = _c(x_f32, np.float32)
    Wgu = _c(Wgu, np.float32)
    Wd = _c(Wd, np.float32)
    H, I = Wd.shape
    gu = np.empty((2 * I,), dtype=np.float32)
    h = np.empty((I,), dtype=np.float32)
    y = np.empty((H,), dtype=np.float32)
    lib().orc_expert_dense(H, I, _p(x), _p(Wgu), _p(Wd), _p(gu), _p(h), _p(y))
    return h, y


def moe_forward(dims, layer: dict, x, ids=None, w=None, nthreads: int = 0,
                want_y: bool = False, want_h: bool = False, want_shared: bool = False):
    """The whole layer on bf16 input x [T][H].  With ids/w given the routing
    is forced; otherwise the oracle routes.  Returns a dict with out (fp32
    [T][H]), ids, w, gap (None when forced), sig, logits (when routed) and,
    on request, y [T][K][H], h [T][K][I], shared [T][H]."""
    H, E, K, I, Is = dims.hidden, dims.n_experts, dims.top_k, dims.inter, dims.shared_inter
    x = _c(x, np.uint16)
    T = x.shape[0]
    keep = {k: (None if v is None else np.ascontiguousarray(v)) for k, v in layer.items()}
    L = OrcLayer(*[_p(keep[n]) for n in (
        "router", "router_bias", "gu_q", "gu_s", "dn_q", "dn_s",
        "sh_gu_q", "sh_gu_s", "sh_dn_q", "sh_dn_s")])
    force = ids is not None
    ids_a = _c(ids, np.int32).copy() if force else np.empty((T, K), dtype=np.int32)
    w_a = _c(w, np.float32).copy() if force else np.empty((T, K), dtype=np.float32)
    gap = None if force else np.empty((T,), dtype=np.float32)
    logits = None if force else np.empty((T, E), dtype=np.float32)
    sig = np.empty((T,), dtype=np.float32)
    out = np.empty((T, H), dtype=np.float32)
    y = np.empty((T, K, H), dtype=np.float32) if want_y else None
    h = np.empty((T, K, I), dtype=np.float32) if want_h else None
    sh = np.empty((T, H), dtype=np.float32) if want_shared else None
    rc = lib().orc_moe_forward(H, E, K, I, Is, ctypes.byref(L), T, _p(x), int(force),
                               _p(ids_a), _p(w_a), _p(gap), _p(sig), _p(out), _p(y), _p(h),
                               _p(sh), _p(logits), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: forced expert id out of range")
    return {"out": out, "ids": ids_a, "w": w_a, "gap": gap, "sig": sig, "logits": logits,
            "y": y, "h": h, "shared": sh}


def stack_forward(dims, layers, r0, forced=None, eps: float = 1e-6, nthreads: int = 0):
    """The residual MoE stack: for each layer l,
         x = bf16(rmsnorm(r)); out = layer_l(x) rounded to bf16; r += out.
    `forced` is an optional list of (ids, w) per layer.  Returns the final
    residual (fp32) and the per-layer records (ids, w, gap, out bf16)."""
    r = _c(r0, np.float32).copy()
    recs = []
    for li, layer in enumerate(layers):
        x = rmsnorm(r, eps)
        if forced is not None:
            res = moe_forward(dims, layer, x, ids=forced[li][0], w=forced[li][1],
                              nthreads=nthreads)
        else:
            res = moe_forward(dims, layer, x, nthreads=nthreads)
        ob = round_bf16(res["out"])
        r = r + bf16_array_to_f32(ob)
        recs.append({"ids": res["ids"], "w": res["w"], "gap": res["gap"], "out_bf16": ob,
                     "x": x})
    return r, recs

"""The C ABI library: it builds, loads, exports every symbol the header
declares, and rejects bad arguments on the host (no GPU needed: validation
happens before any CUDA call)."""
import ctypes
import os
import re

import pytest

import quantized_moe_expert_fwd_gb300 as q
from quantized_moe_expert_fwd_gb300 import build as qbuild
from quantized_moe_expert_fwd_gb300 import pack
from workloads import gen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return q.load()


def _header_functions():
    with open(os.path.join(ROOT, "include", "strata_moe.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"STRATA_API\s+[\w\s\*]+?\b((?:moe|strata)_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _header_functions()
    for n in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_layer_forward",
              "moe_workspace_bytes", "moe_get_device_status", "strata_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _header_functions():
        assert hasattr(lib, n), n
    assert set(_header_functions()) == set(q.strata_moe.EXPORTED)


def _header_arity():
    """Parameter count of every declared prototype (void-parameter lists: 0)."""
    with open(os.path.join(ROOT, "include", "strata_moe.h")) as f:
        text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
    out = {}
    for m in re.finditer(r"STRATA_API\s+[\w\s\*]+?\b((?:moe|strata)_\w+)\s*\(([^)]*)\)", text):
        params = m.group(2).strip()
        out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_signatures_match_the_header(lib):
    """The binding's ctypes argument lists have the header's arity, so a
    changed prototype cannot be called with a stale argument list."""
    arity = _header_arity()
    assert set(arity) == set(_header_functions())
    for name, n in arity.items():
        assert len(getattr(lib, name).argtypes) == n, name


def test_workspace_bytes(lib):
    assert q.moe_workspace_bytes(gen.QWEN, 1) > 0
    assert q.moe_workspace_bytes(gen.QWEN, 32) > q.moe_workspace_bytes(gen.QWEN, 1)
    assert q.moe_workspace_bytes(gen.QWEN, 0) == 0
    bad = gen.LayerDims(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512,
                        group=16)
    assert q.moe_workspace_bytes(bad, 1) == 0
    for kw in ({"hidden": 2000}, {"inter": 384}, {"top_k": 17}, {"n_experts": 4, "top_k": 8},
               {"n_experts": 2048}):
        d = dict(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512)
        d.update(kw)
        assert q.moe_workspace_bytes(gen.LayerDims(**d), 1) == 0, kw


def test_status_strings(lib):
    for s in range(7):
        assert q.strata_status_str(s).startswith("STRATA_")
    assert q.strata_status_str(q.STRATA_ERANGE).startswith("STRATA_ERANGE")
    assert q.strata_status_str(7).startswith("unknown")


def test_invalid_arguments_return_einval_without_launching(lib):
    d = q.strata_moe.dims_struct(gen.QWEN)
    L = q.strata_moe.LayerPtrs()
    null = ctypes.c_void_p(0)
    # NULL layer planes / buffers: rejected on the host
    st = lib.moe_layer_forward(ctypes.byref(d), ctypes.byref(L), null, 1, null, null, null,
                               null, null, 0, null)
    assert st == q.STRATA_EINVAL
    st = lib.moe_route(ctypes.byref(d), ctypes.byref(L), null, 1, null, null, null, null, null,
                       0, null)
    assert st == q.STRATA_EINVAL
    # negative T
    st = lib.moe_permute(ctypes.byref(d), null, -1, null, null, null, null, null, 0, null)
    assert st == q.STRATA_EINVAL
    # T == 0 is a no-op even with NULL buffers once the shape and planes are valid
    st = lib.moe_permute(ctypes.byref(d), null, 0, null, null, null, null, null, 0, null)
    assert st == q.STRATA_OK
    st = lib.moe_rmsnorm(null, 3, 2050, ctypes.c_float(1e-6), null, null)
    assert st == q.STRATA_EINVAL
    # tail-skip: a negative place, and forced ids without forced weights
    st = lib.moe_layer_forward_tail_skip(ctypes.byref(d), ctypes.byref(L), null, 1, -1, null,
                                         null, null, null, null, null, null, 0, null)
    assert st == q.STRATA_EINVAL
    st = lib.moe_layer_forward_tail_skip(ctypes.byref(d), ctypes.byref(L), null, 1, 5,
                                         ctypes.c_void_p(256), null, null, null, null, null, null,
                                         0, null)
    assert st == q.STRATA_EINVAL
    # misaligned workspace pointer
    st = lib.moe_get_device_status(ctypes.c_void_p(8), null)
    assert st == q.STRATA_EINVAL


def test_pack_hand_computed_bytes():
    # (7, -8) -> nibbles (15, 0) -> byte 0x0F ; (0, 0) -> 0x88 ; (-8, 0) -> 0x80 ; (2, -1) -> 0x7A
    q4 = [[7, -8, 0, 0, -8, 0, 2, -1]]
    assert list(pack.pack_int4(q4)[0]) == [0x0F, 0x88, 0x80, 0x7A]
    assert pack.unpack_int4(pack.pack_int4(q4)).tolist() == q4


def test_pack_round_trip_and_interleave():
    import numpy as np
    rng = np.random.default_rng(0)
    qg = rng.integers(-8, 8, (4, 64)).astype(np.int8)
    qu = rng.integers(-8, 8, (4, 64)).astype(np.int8)
    sg = np.full((4, 2), 0.5, dtype=np.float16)
    su = np.full((4, 2), 2.0, dtype=np.float16)
    gq, gs = pack.pack_gate_up(qg, sg, qu, su)
    un = pack.unpack_int4(gq)
    assert np.array_equal(un[0::2], qg) and np.array_equal(un[1::2], qu)
    assert np.all(gs[0::2] == 0x3800) and np.all(gs[1::2] == 0x4000)
    with pytest.raises(ValueError):
        pack.pack_int4([[8, 0]])


def test_phase_trace_needs_the_traced_build(lib):
    """The default library records no phase stamps: a read returns
    STRATA_EUNSUPPORTED (no device call), a NULL buffer STRATA_EINVAL."""
    buf = (ctypes.c_uint64 * 64)()
    assert lib.strata_px_trace_read(ctypes.c_void_p(0), 512) == q.STRATA_EINVAL
    assert lib.strata_px_trace_read(buf, 0) == q.STRATA_EINVAL
    assert lib.strata_px_trace_read(buf, ctypes.sizeof(buf)) == q.STRATA_EUNSUPPORTED

"""moe_layer_forward_static: the layer forward for callers that cannot
allocate device memory (a plugin whose host framework owns all device
allocations, a serving path that must not call cudaMalloc).  It runs on a
fixed workspace inside the library instead of one the caller passes.

Checked through the C ABI against moe_layer_forward with a caller-allocated
workspace, on two calls in a row (the second one reuses the array the first
one left behind), within the tolerance of the other GPU tests; around the
second call the device's free memory (cudaMemGetInfo) and torch's allocated
bytes stay exactly as they were.  This file is
collected last so that a run stopping at its first failure has run every
other test already; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import quantized_moe_expert_fwd_gb300 as q
from tests import gpu_util as G
from workloads import gen

pytestmark = pytest.mark.gpu


def _call_static(lib, dims, dl, x, out):
    d = q.strata_moe.dims_struct(dims)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.moe_layer_forward_static(ctypes.byref(d), ctypes.byref(dl.ptrs),
                                        ctypes.c_void_p(x.data_ptr()), x.shape[0], None, None,
                                        None, ctypes.c_void_p(out.data_ptr()), stream)


def test_static_workspace_matches_caller_workspace_twice():
    q.build.build()
    lib = q.load()
    dims = gen.QWEN
    planes = gen.draw_layer(dims, 31)
    dl = q.DeviceLayer(planes, G.dev())
    for call, T in enumerate((4, 1)):
        xb = oracle.rmsnorm(gen.draw_tokens(dims, T, 300 + call, "resid"))
        x = G.u16(xb)
        want = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
        ws = q.make_workspace(dims, T, G.dev())
        q.moe_layer_forward(dims, dl, x, want, ws)
        got = torch.full((T, dims.hidden), -1, dtype=torch.int16, device=G.dev())
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        held0 = torch.cuda.memory_allocated()
        assert _call_static(lib, dims, dl, x, got) == q.STRATA_OK
        torch.cuda.synchronize()
        if call > 0:
            # the second call: the array and its kernels are in place, and
            # neither the device's free memory nor torch's allocator moved
            assert torch.cuda.mem_get_info()[0] == free0
            assert torch.cuda.memory_allocated() == held0
        g, w = G.bf16_to_np(got), G.bf16_to_np(want)
        G.assert_close(g, w, f"static workspace, call {call + 1}")
        assert q.moe_get_device_status(ws) == q.STRATA_OK


def test_static_workspace_rejects_oversize_requests():
    lib = q.load()
    dims = gen.QWEN
    dl = q.DeviceLayer(gen.draw_layer(dims, 32), G.dev())
    T = q.moe_decode_max_tokens() + 1
    x = torch.zeros((T, dims.hidden), dtype=torch.int16, device=G.dev())
    out = torch.empty((T, dims.hidden), dtype=torch.int16, device=G.dev())
    assert _call_static(lib, dims, dl, x, out) == q.STRATA_EINVAL

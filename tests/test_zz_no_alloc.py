"""The allocation-free decode entry point, moe_layer_forward_decode_noalloc.

It exists for callers that cannot allocate device memory when they run the layer (an engine
whose memory planner owns all of HBM from start-up, a decode loop that must never enter
cudaMalloc/cudaFree, a host program holding only pointers).  Its scratch is a device array owned
by the library.  These tests call it through the C ABI and compare it with moe_layer_forward
(the workspace entry point) on the same token, on two calls in a row, because the array keeps
the previous call's contents.  Both run the same deterministic decode kernel on the same inputs,
so the outputs must agree bit for bit: a stale partial or an arrival counter left over from the
previous call would show.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import bit_quantized_expert_gb300 as moe
import synth

pytestmark = pytest.mark.gpu

def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


@pytest.fixture(scope="module")
def decode_layer():
    from bit_quantized_expert_gb300 import build
    build.build()
    moe.load_library()
    wl = synth.Workload("noalloc_decode", T=1, d=2048, E=64, k=8, F=512, F_shared=512)
    host = synth.make_layer(wl)
    return wl, moe.to_device_layer(host)


def test_noalloc_matches_workspace_entry_point_twice(decode_layer):
    wl, dl = decode_layer
    dm = moe.dims(1, wl.d, wl.E, wl.k, wl.F, wl.F_shared)
    ws = moe.alloc_workspace(dm)
    for seed in (21, 22):                       # two calls in a row on different tokens
        inp = synth.make_inputs(wl, seed=seed)
        x, lg = _dev(inp["x"]), _dev(inp["logits"])
        y_ws = torch.empty((1, wl.d), dtype=torch.float32, device="cuda")
        y_na = torch.full((1, wl.d), float("nan"), dtype=torch.float32, device="cuda")
        moe.layer_forward(dm, x, lg, dl["routed"], dl["shared"], dl["w_sg"], y_ws, ws)
        assert moe.read_error_flags(ws) == 0
        moe.layer_forward_decode_noalloc(dm, x, lg, dl["routed"], dl["shared"], dl["w_sg"], y_na)
        torch.cuda.synchronize()
        a, b = y_na.cpu().numpy(), y_ws.cpu().numpy()
        assert np.isfinite(a).all()
        assert np.array_equal(a, b)


def test_noalloc_rejects_sizes_beyond_its_scratch(decode_layer):
    wl, dl = decode_layer
    lib = moe.load_library()
    re_ = moe.experts_struct(dl["routed"])
    se_ = moe.experts_struct(dl["shared"])
    x = torch.zeros((2, wl.d), dtype=torch.int16, device="cuda")
    lg = torch.zeros((2, wl.E), dtype=torch.float32, device="cuda")
    y = torch.zeros((2, wl.d), dtype=torch.float32, device="cuda")

    def call(dm):
        return lib.moe_layer_forward_decode_noalloc(ctypes.byref(dm), x.data_ptr(), lg.data_ptr(), ctypes.byref(re_),
                                                    ctypes.byref(se_), dl["w_sg"].data_ptr(), y.data_ptr(),
                                                    torch.cuda.current_stream().cuda_stream)

    invalid, unsupported = 1, 2
    assert call(moe.dims(2, wl.d, wl.E, wl.k, wl.F, wl.F_shared)) == unsupported       # more than one token
    # 9 slots x 16 clusters x 16 slices x 128 rows = 294912 partial floats: beyond the 131072 of the array
    assert call(moe.dims(1, wl.d, wl.E, 8, 2048, 2048)) == unsupported
    assert call(moe.dims(0, wl.d, wl.E, wl.k, wl.F, wl.F_shared)) == 0                  # no token: no-op
    # the dims rules of moe_layer_forward, with its status codes
    assert call(moe.dims(1, wl.d + 64, wl.E, wl.k, wl.F, wl.F_shared)) == unsupported   # d % 128 != 0
    assert call(moe.dims(1, wl.d, 2048, wl.k, wl.F, wl.F_shared)) == unsupported       # E > 1024
    assert call(moe.dims(1, wl.d, wl.E, 33, wl.F, wl.F_shared)) == unsupported         # k > 32
    assert call(moe.dims(1, wl.d, wl.E, wl.k, wl.F, 256)) == unsupported               # F_shared != F
    assert call(moe.dims(1, wl.d, wl.E, wl.E + 1, wl.F, wl.F_shared)) == invalid       # k > E
    assert call(moe.dims(-1, wl.d, wl.E, wl.k, wl.F, wl.F_shared)) == invalid          # T < 0

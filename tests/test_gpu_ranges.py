"""Operand-range edges of the two compute paths, against the exact oracle.

The grouped-GEMM path (more than eight tokens) multiplies fp16 operands: x, the dequantised weights
w = q * s + b, and h.  Values above fp16's range (65504) and blocks of values that sit in fp16's
subnormal range (a token whose largest |x|, or a weight row whose largest |w|, is below 2^-12) set
bit 2 of the workspace's error word, and so does a token whose h = silu(x Wg^T) * (x Wu^T) falls
into the subnormal range (small activations with small weights); the caller checks the word with
moe_read_error_flags.  A few tiny
weight rows among normal ones barely move a layer's output, and the layer stays within the exact
bar.  The decode path (up to eight tokens) computes in exact integers and fp32 and has no such
edges: it matches the exact oracle at any of these magnitudes and raises no flag.  With bf16
tensor-core operands (moe_layer_forward_opts) the grouped-GEMM path has fp32's exponent range:
the same inputs raise no flag; scaled x stays within the bf16 bar of the exact oracle, and the
weights far above fp16's range match the oracle that rounds the same operands to bf16 (there
bf16's 8 significant bits alone put the oracle itself 8.8e-2 from the exact layer).
"""
import numpy as np
import pytest
import torch

import bit_quantized_expert_gb300 as moe
import synth
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

EXACT_TOL = 2e-3
BF16_EXACT_TOL = 6e-3   # bf16 operands: derived in test_gpu_parity.py
BF16_EMUL_TOL = 4.2e-3
DECODE_TOL = 2e-5
RANGE_FLAG = 2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_quantized_expert_gb300 import build
    build.build()
    moe.load_library()


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    elif a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(a).cuda()


def _rowwise_err(y, ref):
    y = np.asarray(y, dtype=np.float64)
    return float((np.linalg.norm(y - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-300)).max())


def _run(wl, host, x_bits, logits, T, operands="fp16"):
    dl = moe.to_device_layer(host)
    dm = moe.dims(T, wl.d, wl.E, wl.k, wl.F, wl.F_shared)
    ws = moe.alloc_workspace(dm)
    y = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
    moe.layer_forward(dm, _dev(x_bits[:T]), _dev(logits[:T]), dl["routed"], dl["shared"], dl["w_sg"], y, ws,
                      operands=operands)
    return y.cpu().numpy(), moe.read_error_flags(ws)


def _scaled_x(rng, T, d, scale):
    return synth.f32_to_bf16_bits((rng.standard_normal((T, d)) * scale).astype(np.float32))


@pytest.mark.parametrize("scale", [1e5, 1e-2, 1e-6])
def test_out_of_range_x_flags_the_gemm_path_and_decode_stays_exact(scale):
    """x far above fp16's range (up to ~4e5), small enough that h lands in fp16's subnormal range
    (~1e-2 with these weights: h ~ 1e-5), or itself subnormal (~1e-6): the grouped-GEMM call sets
    the range flag; one to three tokens on the decode kernel match the exact oracle."""
    wl = synth.TINY
    host = synth.make_layer(wl)
    rng = np.random.default_rng(17)
    x = _scaled_x(rng, wl.T, wl.d, scale)
    lg = synth.make_logits(rng, wl)
    _, flags = _run(wl, host, x, lg, wl.T)
    assert flags & RANGE_FLAG
    y, flags = _run(wl, host, x, lg, wl.T, operands="bf16")
    assert flags == 0
    assert _rowwise_err(y, O.moe_layer(x, lg, host, wl.k)["y"]) <= BF16_EXACT_TOL
    for T in (1, 3):
        y, flags = _run(wl, host, x, lg, T)
        assert flags == 0
        ref = O.moe_layer(x[:T], lg[:T], host, wl.k)["y"]
        assert _rowwise_err(y, ref) <= DECODE_TOL, T


def test_small_but_normal_x_raises_no_flag():
    """x around 0.25: x and h stay in fp16's normal range, no flag, and the grouped-GEMM layer is
    within the exact bar."""
    wl = synth.TINY
    host = synth.make_layer(wl)
    rng = np.random.default_rng(18)
    x = _scaled_x(rng, wl.T, wl.d, 0.25)
    lg = synth.make_logits(rng, wl)
    y, flags = _run(wl, host, x, lg, wl.T)
    assert flags == 0
    ref = O.moe_layer(x, lg, host, wl.k)["y"]
    assert _rowwise_err(y, ref) <= EXACT_TOL


def _shrink_rows(qm, rows, rng, lo, hi):
    """Scales of the given rows of every expert drawn from [lo, hi] (log-uniform), biases -8 s."""
    s = np.exp(rng.uniform(np.log(lo), np.log(hi), size=qm["scales"][:, rows].shape)).astype(np.float32)
    qm["scales"][:, rows] = synth.f32_to_bf16_bits(s)
    qm["biases"][:, rows] = synth.f32_to_bf16_bits(-8.0 * synth.bf16_bits_to_f32(qm["scales"][:, rows]))


def test_tiny_scale_rows_stay_within_the_exact_bar():
    """A few rows of every gate, up and down matrix with scales and biases between 1e-9 and 1e-6 (their
    weights are fp16 subnormals or zero): those rows add almost nothing to the layer, the
    grouped-GEMM output stays within the exact bar, and the range flag reports the subnormal rows.
    The decode kernel matches the exact oracle and raises no flag."""
    wl = synth.TINY
    host = synth.make_layer(wl, seed=4)
    rng = np.random.default_rng(19)
    for ex in (host["routed"], host["shared"]):
        _shrink_rows(ex["gate"], [3, 50, 127], rng, 1e-9, 1e-6)
        _shrink_rows(ex["up"], [7, 64], rng, 1e-9, 1e-6)
        _shrink_rows(ex["down"], [0, 100, 255], rng, 1e-9, 1e-6)
    inp = synth.make_inputs(wl, seed=6)
    y, flags = _run(wl, host, inp["x"], inp["logits"], wl.T)
    assert flags & RANGE_FLAG
    ref = O.moe_layer(inp["x"], inp["logits"], host, wl.k)["y"]
    assert _rowwise_err(y, ref) <= EXACT_TOL
    for T in (1, 2):
        y, flags = _run(wl, host, inp["x"], inp["logits"], T)
        assert flags == 0
        ref = O.moe_layer(inp["x"][:T], inp["logits"][:T], host, wl.k)["y"]
        assert _rowwise_err(y, ref) <= DECODE_TOL, T


def test_weights_above_fp16_range_flag_the_gemm_path():
    """Scales near 1e4 put 15 |s| + |b| above 65504 in a few rows: the grouped-GEMM call sets the
    range flag; the decode kernel stays exact."""
    wl = synth.TINY
    host = synth.make_layer(wl, seed=5)
    rng = np.random.default_rng(20)
    _shrink_rows(host["routed"]["up"], [9], rng, 8e3, 1.2e4)
    inp = synth.make_inputs(wl, seed=7)
    _, flags = _run(wl, host, inp["x"], inp["logits"], wl.T)
    assert flags & RANGE_FLAG
    y, flags = _run(wl, host, inp["x"], inp["logits"], wl.T, operands="bf16")
    assert flags == 0
    emu = O.moe_layer(inp["x"], inp["logits"], host, wl.k, operands="bf16", out16="bf16")["y"]
    assert _rowwise_err(y, emu) <= BF16_EMUL_TOL
    y, flags = _run(wl, host, inp["x"], inp["logits"], 1)
    assert flags == 0
    ref = O.moe_layer(inp["x"][:1], inp["logits"][:1], host, wl.k)["y"]
    assert _rowwise_err(y, ref) <= DECODE_TOL

"""Grouped-query decode attention on the GPU against the float64 oracle.

Bar (per output element, from the arithmetic): |o - o_ref| <= TOL * mag, where mag[h, :] is the
same attention applied to |V| (the oracle on the values' magnitudes), the scale against which
rounding in a weighted sum is bounded.  The kernel's error sources, relative to mag:
  * p enters the value product as bf16(p) + bf16(p - bf16(p)): at most 2^-17;
  * fp32 accumulation over a CTA's run of tiles and the two fixed-order merges: about 2^-24 per
    step over a few dozen steps;
  * scores in fp32: an absolute error of about 2^-24 * sum_i |q_i k_i| / sqrt(128) in base-2 units,
    which moves p by that fraction; with the inputs here (score spread up to 8) well below 2^-17.
TOL = 2^-16 covers the sum: the P split is at most 2^-17 and the fp32 terms stay below 2^-17 at
these sizes (a few hundred steps at most).  Results must also be identical from call to call.
"""
import numpy as np
import pytest
import torch

import bit_quantized_expert_gb300 as moe
import synth
from oracle import attention_oracle as A

pytestmark = pytest.mark.gpu

TOL = 2.0 ** -16


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_quantized_expert_gb300 import build
    build.build()
    moe.load_library()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _run(Hq, Hkv, N, inp, capacity=None):
    gd = moe.gqa_dims(Hq, Hkv, 128, N, capacity)
    ws = moe.alloc_gqa_workspace(gd)
    o = torch.empty((Hq, 128), dtype=torch.float32, device="cuda")
    moe.gqa_decode_attention(gd, _dev(inp["q"]), _dev(inp["k"]), _dev(inp["v"]), o, ws)
    return o.cpu().numpy().astype(np.float64), moe.read_error_flags(ws)


def _check(o, inp, N, label=""):
    k, v = inp["k"][:, :N], inp["v"][:, :N]
    ref = A.gqa_decode_attention(inp["q"], k, v)
    mag = A.gqa_decode_attention(inp["q"], k, v & np.uint16(0x7FFF))
    ratio = np.abs(o - ref) / np.maximum(mag, 1e-30)
    worst = float(ratio.max())
    print(f"{label} N={N}: max |o - ref| / mag = {worst:.3e} (bar {TOL:.3e})")
    assert worst <= TOL, (label, N, worst)


@pytest.mark.parametrize("N", [1, 37, 64, 65, 1000, 4097, 9000])
def test_small_contexts_sixteen_over_two(N):
    """The model's head shape (16 query heads, 2 key/value heads) from one position to several
    blocks with ragged tails."""
    inp = synth.make_attention(16, 2, 128, N, seed=N)
    o, flags = _run(16, 2, N, inp)
    assert flags == 0
    _check(o, inp, N, "16/2")


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (6, 2), (8, 2), (4, 1), (32, 4), (7, 7)])
def test_group_sizes(Hq, Hkv):
    """Groups of 1, 3, 4, 8 query heads per key/value head and up to eight key/value heads."""
    N = 777
    inp = synth.make_attention(Hq, Hkv, 128, N, seed=Hq * 10 + Hkv)
    o, flags = _run(Hq, Hkv, N, inp)
    assert flags == 0
    _check(o, inp, N, f"{Hq}/{Hkv}")


def test_capacity_beyond_context_is_never_read():
    """A cache allocated for 3000 positions holding NaN patterns past N = 1234: the output is finite
    and matches the oracle on the first N positions."""
    N, cap = 1234, 3000
    inp = synth.make_attention(16, 2, 128, N, capacity=cap, seed=5, tail_bits=0x7FC0)
    o, flags = _run(16, 2, N, inp, capacity=cap)
    assert flags == 0 and np.isfinite(o).all()
    _check(o, inp, N, "capacity")


@pytest.mark.parametrize("q_scale", [8.0, 0.01])
def test_peaked_and_flat_scores(q_scale):
    """Scores with spread 8 (a few positions dominate) and 0.01 (nearly uniform weights)."""
    N = 5000
    inp = synth.make_attention(16, 2, 128, N, seed=7, q_scale=q_scale)
    o, flags = _run(16, 2, N, inp)
    assert flags == 0
    _check(o, inp, N, f"q_scale={q_scale}")


def test_one_dominant_position_returns_its_value():
    """A key equal to a large multiple of the query at one position: that head returns the
    position's value (the other weights are below 2^-100)."""
    N = 3000
    inp = synth.make_attention(16, 2, 128, N, seed=9)
    qf = synth.bf16_bits_to_f32(inp["q"][3])
    inp["k"][0, 1777] = synth.f32_to_bf16_bits(qf * 8.0)
    o, flags = _run(16, 2, N, inp)
    assert flags == 0
    vv = synth.bf16_bits_to_f32(inp["v"][0, 1777]).astype(np.float64)
    assert np.allclose(o[3], vv, rtol=1e-6, atol=1e-6)
    _check(o, inp, N, "dominant")


def test_identical_across_calls():
    N = 20000
    inp = synth.make_attention(16, 2, 128, N, seed=11)
    a, _ = _run(16, 2, N, inp)
    b, _ = _run(16, 2, N, inp)
    assert np.array_equal(a, b)


def test_non_finite_query_sets_the_flag():
    """An infinite query component makes that head's scores infinite: its output is not finite and
    bit 8 of the error word is set."""
    N = 500
    inp = synth.make_attention(16, 2, 128, N, seed=12)
    inp["q"][5, 17] = 0x7F80
    o, flags = _run(16, 2, N, inp)
    assert flags & moe.ERR_NON_FINITE
    assert not np.isfinite(o[5]).all()


@pytest.mark.parametrize("wl", [synth.GQA_32K, synth.GQA_128K], ids=lambda w: w.name)
def test_full_size_context(wl):
    """The pages' context lengths with the model's head shape, every output against the oracle, in
    the launch configuration the benchmark times (one call per layer)."""
    inp = synth.make_attention(wl.Hq, wl.Hkv, wl.D, wl.N, seed=21)
    o, flags = _run(wl.Hq, wl.Hkv, wl.N, inp)
    assert flags == 0
    _check(o, inp, wl.N, wl.name)

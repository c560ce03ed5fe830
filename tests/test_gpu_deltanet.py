"""Gated DeltaNet scan on the GPU against the float64 oracle.

Bar (per element, from the arithmetic): |o_t[i] - ref| <= tol(T) * |S_t[i, :]| / sqrt(128), the
Cauchy-Schwarz scale of o_t[i] = S_t[i, :] . q^_t (|q^_t| <= 1/sqrt(128)), and the same tol(T) on
every final-state element relative to its row norm.  The scan keeps the state in fp32: one token
rounds each state element a few times (a 16-term partial dot, a 3-step butterfly, the update), the
normalisation of k and q in fp32 adds a relative error near 2^-23, and the recurrence does not
amplify errors (|a_t S (I - b_t k k^T)| <= |S|), so rounding accumulates at most linearly in T and
in practice like a random walk.  tol(T) = 2^-20 * (4 + sqrt(T)) allows about sixteen units of
fp32 rounding per step on a random walk.
Splitting a sequence into two calls must give bit-identical results (the state passes through
fp32 memory unchanged), and so must repeating a call.
"""
import math

import numpy as np
import pytest
import torch

import bit_quantized_expert_gb300 as moe
import synth
from oracle import deltanet_oracle as O

pytestmark = pytest.mark.gpu


def tol(T):
    return 2.0 ** -20 * (4.0 + math.sqrt(T))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from bit_quantized_expert_gb300 import build
    build.build()
    moe.load_library()


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def _run(inp, T, H, S=None, in_place=False):
    gd = moe.gdn_dims(T, H)
    ws = moe.alloc_gdn_workspace(gd)
    s_in = _dev(inp["S0"]) if S is None else S
    s_out = s_in if in_place else torch.empty_like(s_in)
    o = torch.empty((max(T, 1), H, 128), dtype=torch.float32, device="cuda")
    moe.gdn_scan(gd, _dev(inp["q"][:T]), _dev(inp["k"][:T]), _dev(inp["v"][:T]), _dev(inp["g"][:T]),
                 _dev(inp["beta"][:T]), s_in, s_out, o, ws)
    return o[:T].cpu().numpy().astype(np.float64), s_out, moe.read_error_flags(ws)


def _check(o, s_out, inp, T, label):
    ref, S_ref, nrm = O.gated_delta_rule(inp["q"][:T], inp["k"][:T], inp["v"][:T], inp["g"][:T], inp["beta"][:T],
                                         inp["S0"], want_row_norms=True)
    scale = np.maximum(nrm / math.sqrt(128), 1e-30)
    r_o = float((np.abs(o - ref) / scale).max())
    S = s_out.cpu().numpy().astype(np.float64)
    r_s = float((np.abs(S - S_ref) / np.maximum(np.sqrt((S_ref ** 2).sum(axis=2, keepdims=True)), 1e-30)).max())
    print(f"{label} T={T}: o {r_o:.3e}, state {r_s:.3e} (bar {tol(T):.3e})")
    assert r_o <= tol(T) and r_s <= tol(T), (label, T, r_o, r_s)


@pytest.mark.parametrize("T,H", [(1, 1), (5, 3), (31, 2), (32, 16), (33, 4), (100, 16), (257, 5)])
def test_small_sequences(T, H):
    """One token to several 32-token chunks with ragged tails, from a non-zero state."""
    inp = synth.make_scan(T, H, 128, seed=T * 7 + H)
    o, s_out, flags = _run(inp, T, H)
    assert flags == 0
    _check(o, s_out, inp, T, f"H={H}")


@pytest.mark.parametrize("wl", [synth.SCAN_512, synth.SCAN_2048], ids=lambda w: w.name)
def test_full_size_prompts(wl):
    """The prompt lengths of the benchmark (fresh state, 16 heads), every output and the final state."""
    inp = synth.make_scan(wl.T, wl.H, wl.D, seed=3, fresh=wl.fresh)
    o, s_out, flags = _run(inp, wl.T, wl.H)
    assert flags == 0
    _check(o, s_out, inp, wl.T, wl.name)


def test_decode_step_in_place():
    """One token per call with the state updated in place, as the decode step runs it."""
    inp = synth.make_scan(3, 16, 128, seed=11)
    S = _dev(inp["S0"])
    outs = []
    for t in range(3):
        one = {key: val[t:t + 1] for key, val in inp.items() if key != "S0"}
        o, S, flags = _run(one, 1, 16, S=S, in_place=True)
        assert flags == 0
        outs.append(o[0])
    _check(np.stack(outs), S, inp, 3, "decode")


def test_early_state_read_is_bit_identical():
    """GDN_OPT_STATE_EARLY only moves the state load ahead of the dependency wait: a decode loop over
    several layers, each with its own state updated in place, gives the same bits with and without
    it."""
    H, layers, steps = 16, 3, 4
    inps = [synth.make_scan(steps, H, 128, seed=60 + l) for l in range(layers)]
    gd = moe.gdn_dims(1, H)
    ws = moe.alloc_gdn_workspace(gd)
    outs = {}
    for early in (False, True):
        S = [_dev(inp["S0"]) for inp in inps]
        o = torch.empty((1, H, 128), dtype=torch.float32, device="cuda")
        got = []
        for t in range(steps):
            for l, inp in enumerate(inps):
                one = {key: _dev(np.ascontiguousarray(val[t:t + 1])) for key, val in inp.items() if key != "S0"}
                moe.gdn_scan(gd, one["q"], one["k"], one["v"], one["g"], one["beta"], S[l], S[l], o, ws,
                             early_state=early)
                got.append(o.cpu().numpy().copy())
        outs[early] = (got, [s_.cpu().numpy() for s_ in S])
    assert moe.read_error_flags(ws) == 0
    assert all(np.array_equal(a, b) for a, b in zip(outs[False][0], outs[True][0]))
    assert all(np.array_equal(a, b) for a, b in zip(outs[False][1], outs[True][1]))


def test_split_calls_are_bit_identical():
    """150 tokens in one call, and as 100 then 50 tokens with the state passed on: identical bits
    (every token's arithmetic is the same and the state passes through fp32 memory unchanged); a
    repeated call is identical too."""
    T, H = 150, 4
    inp = synth.make_scan(T, H, 128, seed=21)
    o_all, s_all, _ = _run(inp, T, H)
    o_rep, s_rep, _ = _run(inp, T, H)
    first = {key: val[:100] for key, val in inp.items() if key != "S0"}
    first["S0"] = inp["S0"]
    o1, s1, _ = _run(first, 100, H)
    second = {key: val[100:] for key, val in inp.items() if key != "S0"}
    o2, s2, flags = _run(second, 50, H, S=s1)
    assert flags == 0
    assert np.array_equal(o_all, np.concatenate([o1, o2]))
    assert torch.equal(s_all, s2) and torch.equal(s_all, s_rep) and np.array_equal(o_all, o_rep)


@pytest.mark.parametrize("T", [63, 64, 65, 95, 96, 97])
def test_lengths_around_staging_chunks(T):
    """Lengths on both sides of two and three 32-token staging chunks, from a non-zero state."""
    inp = synth.make_scan(T, 3, 128, seed=T)
    o, s_out, flags = _run(inp, T, 3)
    assert flags == 0
    _check(o, s_out, inp, T, "chunks")


def test_strong_decay_and_repeated_keys():
    """Decay down to 0.05 per token and a run of twenty identical keys written with strength 0.99:
    still within the bar."""
    T, H = 192, 2
    inp = synth.make_scan(T, H, 128, seed=23)
    rng = np.random.default_rng(24)
    inp["g"] = np.log(rng.uniform(0.05, 1.0, (T, H))).astype(np.float32)
    inp["k"][10:30] = inp["k"][10]
    inp["beta"][10:30] = 0.99
    o, s_out, flags = _run(inp, T, H)
    assert flags == 0
    _check(o, s_out, inp, T, "strong decay")


def test_zero_keys_only_decay():
    """Tokens whose key is all zeros write nothing (k^ = 0): the state only decays."""
    T, H = 40, 2
    inp = synth.make_scan(T, H, 128, seed=31)
    inp["k"][5:20] = 0
    o, s_out, flags = _run(inp, T, H)
    assert flags == 0
    _check(o, s_out, inp, T, "zero keys")


def test_empty_sequence_copies_the_state():
    inp = synth.make_scan(1, 16, 128, seed=41)
    gd = moe.gdn_dims(0, 16)
    ws = moe.alloc_gdn_workspace(gd)
    s_in = _dev(inp["S0"])
    s_out = torch.zeros_like(s_in)
    dummy = torch.zeros(16, dtype=torch.float32, device="cuda")
    moe.gdn_scan(gd, dummy, dummy, dummy, dummy, dummy, s_in, s_out, dummy, ws)
    torch.cuda.synchronize()
    assert torch.equal(s_in, s_out)


def test_non_finite_state_sets_the_flag():
    inp = synth.make_scan(4, 2, 128, seed=51)
    inp["S0"][1, 7, 3] = np.inf
    _, _, flags = _run(inp, 4, 2)
    assert flags & moe.ERR_NON_FINITE

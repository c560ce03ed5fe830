"""Pins of the grouped-query decode attention oracle against facts fixed outside it: closed forms,
the head-to-group map, exact reductions and a pure-Python brute force.  No GPU needed.

Each pin targets a plausible oracle mistake: a wrong softmax axis, a missing or wrong 1/sqrt(D)
scale, query heads mapped to the wrong key/value head (h % Hkv instead of h // group), K and V
swapped, a transposed cache."""
import math

import numpy as np

import synth
from oracle import attention_oracle as A


def _bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_equal_scores_average_the_values():
    """All keys zero: every score is equal, so each head returns the mean of its group's values."""
    rng = np.random.default_rng(1)
    Hq, Hkv, D, N = 8, 2, 16, 9
    q = _bits(rng.standard_normal((Hq, D)))
    k = _bits(np.zeros((Hkv, N, D)))
    v = _bits(rng.standard_normal((Hkv, N, D)))
    o = A.gqa_decode_attention(q, k, v)
    vv = A.bf16_to_f64(v)
    for h in range(Hq):
        assert np.allclose(o[h], vv[h // 4].mean(axis=0), rtol=1e-14, atol=1e-15)


def test_single_position_returns_its_value():
    rng = np.random.default_rng(2)
    q = _bits(rng.standard_normal((4, 8)))
    k = _bits(rng.standard_normal((2, 1, 8)))
    v = _bits(rng.standard_normal((2, 1, 8)))
    o = A.gqa_decode_attention(q, k, v)
    vv = A.bf16_to_f64(v)
    assert np.array_equal(o, np.repeat(vv[:, 0], 2, axis=0))


def test_heads_read_their_own_group():
    """Group 0's values are 1 and group 1's are 2: query heads 0..7 must return 1, heads 8..15 must
    return 2 (a map by h % Hkv would interleave them)."""
    rng = np.random.default_rng(3)
    Hq, Hkv, D, N = 16, 2, 128, 5
    q = _bits(rng.standard_normal((Hq, D)))
    k = _bits(rng.standard_normal((Hkv, N, D)))
    v = _bits(np.stack([np.ones((N, D)), 2 * np.ones((N, D))]))
    o = A.gqa_decode_attention(q, k, v)
    assert np.allclose(o[:8], 1.0, rtol=1e-14) and np.allclose(o[8:], 2.0, rtol=1e-14)


def test_two_positions_closed_form_with_the_scale():
    """Two positions whose keys differ only along the query: the weight of position 1 is the logistic
    of the score gap (q . (k1 - k0)) / sqrt(D).  Keys as K and values as V: swapping them changes the
    result."""
    D = 64
    q = np.zeros((1, D))
    q[0, 0] = 2.0
    k = np.zeros((1, 2, D))
    k[0, 1, 0] = 3.0            # score gap 6 / 8 = 0.75
    v = np.zeros((1, 2, D))
    v[0, 0, 1] = 1.0
    v[0, 1, 2] = 1.0
    o = A.gqa_decode_attention(_bits(q), _bits(k), _bits(v))
    w1 = 1.0 / (1.0 + math.exp(-6.0 / math.sqrt(D)))
    assert abs(o[0, 2] - w1) < 1e-15 and abs(o[0, 1] - (1.0 - w1)) < 1e-15
    assert np.all(o[0, 3:] == 0.0) and o[0, 0] == 0.0


def test_bruteforce_python_tiny():
    """Plain Python loops with math.exp on a tiny case (2 groups of 3 heads, 7 positions)."""
    rng = np.random.default_rng(4)
    Hq, Hkv, D, N = 6, 2, 8, 7
    q = _bits(rng.standard_normal((Hq, D)) * 2)
    k = _bits(rng.standard_normal((Hkv, N, D)))
    v = _bits(rng.standard_normal((Hkv, N, D)))
    got = A.gqa_decode_attention(q, k, v)
    qf, kf, vf = A.bf16_to_f64(q), A.bf16_to_f64(k), A.bf16_to_f64(v)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = [sum(float(qf[h, c]) * float(kf[g, n, c]) for c in range(D)) / math.sqrt(D) for n in range(N)]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        want = [sum(e[n] * float(vf[g, n, c]) for n in range(N)) / sum(e) for c in range(D)]
        assert np.allclose(got[h], want, rtol=1e-12, atol=1e-14)


def test_position_order_does_not_matter():
    """Attention is a sum over positions: permuting the cache's positions (keys and values
    together) leaves the output unchanged."""
    rng = np.random.default_rng(5)
    q = _bits(rng.standard_normal((4, 32)))
    k = _bits(rng.standard_normal((2, 50, 32)))
    v = _bits(rng.standard_normal((2, 50, 32)))
    perm = rng.permutation(50)
    a = A.gqa_decode_attention(q, k, v)
    b = A.gqa_decode_attention(q, k[:, perm], v[:, perm])
    assert np.allclose(a, b, rtol=1e-13, atol=1e-15)


def test_large_scores_do_not_overflow():
    """Scores of several thousand (far beyond exp's range): the result is the value of the single
    highest-scoring position, finite, as the softmax's definition gives."""
    D, N = 64, 6
    q = np.zeros((1, D))
    q[0, 0] = 256.0
    k = np.zeros((1, N, D))
    k[0, :, 0] = 128.0
    k[0, 3, 0] = 256.0                      # score 8192 against 4096 for the others
    rng = np.random.default_rng(6)
    v = rng.standard_normal((1, N, D))
    o = A.gqa_decode_attention(_bits(q), _bits(k), _bits(v))
    assert np.isfinite(o).all()
    assert np.array_equal(o[0], A.bf16_to_f64(_bits(v))[0, 3])

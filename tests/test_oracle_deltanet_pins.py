"""Pins of the Gated DeltaNet oracle against facts fixed outside it: closed forms of the decay and
of the delta-rule write, the defining property of the delta rule, orthogonal keys, a pure-Python
brute force and head independence.  No GPU needed.

Each pin targets a plausible mistake: the decay applied after the write or not at all, the write
using the decayed or the undecayed state the wrong way round, k and v swapped in the outer
product, a missing 1/sqrt(Dk) on q, a missing normalisation of k, heads mixed."""
import math

import numpy as np

import synth
from oracle import deltanet_oracle as O


def _bits(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))


def _inputs(rng, T, H, D, S0_scale=0.3):
    q = _bits(rng.standard_normal((T, H, D)))
    k = _bits(rng.standard_normal((T, H, D)))
    v = _bits(rng.standard_normal((T, H, D)))
    g = np.log(rng.uniform(0.8, 0.999, (T, H))).astype(np.float32)
    beta = rng.uniform(0.05, 0.95, (T, H)).astype(np.float32)
    S0 = (rng.standard_normal((H, D, D)) * S0_scale).astype(np.float32)
    return q, k, v, g, beta, S0


def test_no_write_is_pure_decay():
    """beta = 0: S_t = exp(g_1 + .. + g_t) S_0 and o_t = S_t q_t-hat."""
    rng = np.random.default_rng(1)
    T, H, D = 5, 2, 8
    q, k, v, g, beta, S0 = _inputs(rng, T, H, D)
    beta[:] = 0
    o, ST = O.gated_delta_rule(q, k, v, g, beta, S0)
    qf = synth.bf16_bits_to_f32(q).astype(np.float64)
    for h in range(H):
        decay = np.exp(np.cumsum(g[:, h].astype(np.float64)))
        assert np.allclose(ST[h], decay[-1] * S0[h], rtol=1e-12, atol=0)
        for t in range(T):
            qhat = qf[t, h] / math.sqrt((qf[t, h] ** 2).sum() + 1e-6) / math.sqrt(D)
            assert np.allclose(o[t, h], decay[t] * (S0[h].astype(np.float64) @ qhat), rtol=1e-11, atol=1e-14)


def test_single_write_from_zero_state():
    """S_0 = 0, g = 0, beta = 1, k = 3 e_2, q = 2 e_2: S_1 = v k-hat^T and
    o = v * (3 / sqrt(9 + 1e-6)) * (2 / sqrt(4 + 1e-6)) / sqrt(D)."""
    D = 16
    q = np.zeros((1, 1, D)); q[0, 0, 2] = 2.0
    k = np.zeros((1, 1, D)); k[0, 0, 2] = 3.0
    rng = np.random.default_rng(2)
    v = _bits(rng.standard_normal((1, 1, D)))
    o, ST = O.gated_delta_rule(_bits(q), _bits(k), v, np.zeros((1, 1), np.float32), np.ones((1, 1), np.float32),
                               np.zeros((1, D, D), np.float32))
    vf = synth.bf16_bits_to_f32(v[0, 0]).astype(np.float64)
    kn = 3.0 / math.sqrt(9.0 + 1e-6)
    assert np.allclose(o[0, 0], vf * kn * (2.0 / math.sqrt(4.0 + 1e-6)) / math.sqrt(D), rtol=1e-14, atol=0)
    want = np.zeros((D, D)); want[:, 2] = vf * kn
    assert np.allclose(ST[0], want, rtol=1e-14, atol=0)


def test_full_write_maps_the_key_to_its_value():
    """Delta rule with beta = 1 and no decay: after a token, the state sends that token's
    (normalised) key to its value, S_t k_t = v_t, whatever the state before.  Keys of norm ~100 make
    the 1e-6 in the normalisation negligible."""
    rng = np.random.default_rng(3)
    T, H, D = 4, 3, 32
    q, _, v, g, beta, S0 = _inputs(rng, T, H, D)
    k = _bits(rng.standard_normal((T, H, D)) * 20.0)
    g[:] = 0
    beta[:] = 1
    for t_end in range(1, T + 1):
        _, ST = O.gated_delta_rule(q[:t_end], k[:t_end], v[:t_end], g[:t_end], beta[:t_end], S0)
        kf = synth.bf16_bits_to_f32(k[t_end - 1]).astype(np.float64)
        vf = synth.bf16_bits_to_f32(v[t_end - 1]).astype(np.float64)
        for h in range(H):
            khat = kf[h] / np.linalg.norm(kf[h])
            assert np.allclose(ST[h] @ khat, vf[h], rtol=1e-8, atol=1e-8)


def test_orthogonal_keys_closed_form():
    """Token t writes along basis direction j_t (distinct), no decay: column j_t of the final state
    is (1 - b_t) S_0[:, j_t] + b_t v_t and every other column keeps S_0's."""
    rng = np.random.default_rng(4)
    T, H, D = 6, 1, 16
    q, _, v, g, beta, S0 = _inputs(rng, T, H, D)
    cols = [5, 0, 11, 3, 15, 8]
    k = np.zeros((T, H, D))
    for t, j in enumerate(cols):
        k[t, 0, j] = 100.0
    g[:] = 0
    _, ST = O.gated_delta_rule(q, _bits(k), v, g, beta, S0)
    vf = synth.bf16_bits_to_f32(v).astype(np.float64)
    want = S0[0].astype(np.float64).copy()
    for t, j in enumerate(cols):
        b = float(beta[t, 0])
        want[:, j] = (1.0 - b) * S0[0][:, j].astype(np.float64) + b * vf[t, 0]
    assert np.allclose(ST[0], want, rtol=1e-9, atol=1e-9)


def test_bruteforce_python_tiny():
    """Scalar Python loops with math.exp and explicit sums on 2 heads, 3 tokens, size 4."""
    rng = np.random.default_rng(5)
    T, H, D = 3, 2, 4
    q, k, v, g, beta, S0 = _inputs(rng, T, H, D)
    o, ST = O.gated_delta_rule(q, k, v, g, beta, S0)
    qf, kf, vf = (synth.bf16_bits_to_f32(a).astype(np.float64) for a in (q, k, v))
    for h in range(H):
        S = [[float(S0[h, i, j]) for j in range(D)] for i in range(D)]
        for t in range(T):
            kn = math.sqrt(sum(x * x for x in kf[t, h]) + 1e-6)
            qn = math.sqrt(sum(x * x for x in qf[t, h]) + 1e-6) * math.sqrt(D)
            kh = [x / kn for x in kf[t, h]]
            qh = [x / qn for x in qf[t, h]]
            a = math.exp(float(g[t, h]))
            b = float(beta[t, h])
            for i in range(D):
                sk = sum(S[i][j] * kh[j] for j in range(D))          # S_{t-1} k
                c = b * (float(vf[t, h, i]) - a * sk)
                S[i] = [a * S[i][j] + c * kh[j] for j in range(D)]
                assert abs(sum(S[i][j] * qh[j] for j in range(D)) - o[t, h, i]) < 1e-12
        assert np.allclose(ST[h], np.array(S), rtol=1e-12, atol=1e-13)


def test_heads_are_independent():
    """Permuting the heads of every input permutes the outputs and states the same way."""
    rng = np.random.default_rng(6)
    T, H, D = 4, 5, 8
    q, k, v, g, beta, S0 = _inputs(rng, T, H, D)
    perm = np.array([3, 0, 4, 1, 2])
    o, ST = O.gated_delta_rule(q, k, v, g, beta, S0)
    o2, ST2 = O.gated_delta_rule(q[:, perm], k[:, perm], v[:, perm], g[:, perm], beta[:, perm], S0[perm])
    assert np.allclose(o2, o[:, perm], rtol=1e-14, atol=0) and np.allclose(ST2, ST[perm], rtol=1e-14, atol=0)


def test_row_norms_are_those_of_the_state():
    rng = np.random.default_rng(7)
    q, k, v, g, beta, S0 = _inputs(rng, 3, 2, 8)
    o, ST, nrm = O.gated_delta_rule(q, k, v, g, beta, S0, want_row_norms=True)
    assert np.allclose(nrm[-1], np.sqrt((ST ** 2).sum(axis=2)), rtol=1e-14)

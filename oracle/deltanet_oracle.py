"""CPU oracle for the Gated DeltaNet recurrence (the model's thirty recurrent layers).

TEST INFRASTRUCTURE ONLY.  This module is the plain float64 statement of what the recurrent scan
computes.  Only the test suite, the package smoke check and the CPU-baseline leg of the benchmark
may import it; the CUDA library never does and shares no code with it.

Where the pages speak of it: the model mixes thirty Gated DeltaNet layers, a fixed-size
recurrence, into its stack ("Perplexity libera Lily: inferencia en Rust y Metal para Mac",
section "Tres formas de carga en un mismo modelo"); the engine scans that recurrence with the
state carried in registers, which lifted prefill by 5.6 % (same page, section "Prefill: pesos
comprimidos y enrutamiento en la GPU"; "Perplexity ouvre le code de Lily...", lefilia.fr, article
body).  The pages do not print the recurrence.  It is the gated delta rule of the published Gated
DeltaNet (Yang, Kautz and Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule",
ICLR 2025), restated here: per head, a state S of shape [Dv, Dk] evolves as

    S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,     o_t = S_t q_t,

with the decay a_t = exp(g_t) (g_t <= 0) and the write strength b_t in (0, 1).
Readings (the pages are silent): 16 heads with Dk = Dv = 128 (hidden size / heads); q and k are
L2-normalised per head and token, x / sqrt(|x|^2 + 1e-6), and q is further scaled by 1/sqrt(Dk),
as the published layer does; g and b arrive already computed (the gate projections are outside
the scan); bf16 q, k, v; fp32 g, b, initial state; the state and outputs in float64 here.
"""
from __future__ import annotations

import math

import numpy as np

L2_EPS = 1e-6


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def l2_normalise(x: np.ndarray) -> np.ndarray:
    """x / sqrt(sum(x^2) + 1e-6) along the last axis."""
    return x / np.sqrt((x * x).sum(axis=-1, keepdims=True) + L2_EPS)


def gated_delta_rule(q_bits, k_bits, v_bits, g, beta, S0, want_row_norms: bool = False):
    """The recurrence above over T tokens, token by token, for every head.

    q_bits, k_bits  bf16 [T, H, Dk]
    v_bits          bf16 [T, H, Dv]
    g               fp32 [T, H]        log decay (<= 0)
    beta            fp32 [T, H]        write strength
    S0              fp32 [H, Dv, Dk]   state before the first token
    Returns o float64 [T, H, Dv] and the final state float64 [H, Dv, Dk]; with want_row_norms
    also |S_t[i, :]|_2 for every token, head and row (float64 [T, H, Dv]), the scale against
    which the rounding of o_t[i] = S_t[i, :] . q_t is bounded."""
    q = bf16_to_f64(q_bits)
    k = bf16_to_f64(k_bits)
    v = bf16_to_f64(v_bits)
    g = np.asarray(g, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    T, H, Dk = q.shape
    Dv = v.shape[2]
    S_all = np.array(S0, dtype=np.float64).reshape(H, Dv, Dk)
    o = np.zeros((T, H, Dv))
    norms = np.zeros((T, H, Dv)) if want_row_norms else None
    for h in range(H):
        S = S_all[h].copy()
        for t in range(T):
            kt = l2_normalise(k[t, h])
            qt = l2_normalise(q[t, h]) / math.sqrt(Dk)
            S = math.exp(g[t, h]) * S                          # decay
            S = S + beta[t, h] * np.outer(v[t, h] - S @ kt, kt)   # delta-rule write
            o[t, h] = S @ qt
            if want_row_norms:
                norms[t, h] = np.sqrt((S * S).sum(axis=1))
        S_all[h] = S
    if want_row_norms:
        return o, S_all, norms
    return o, S_all

"""CPU oracle for grouped-query decode attention over a KV cache.

TEST INFRASTRUCTURE ONLY.  This module is the plain float64 statement of what the attention
decode step computes.  Only the test suite, the package smoke check and the CPU-baseline leg of
the benchmark may import it; the CUDA library never does and shares no code with it.

What it computes, and where the pages say so:
* The engine's model mixes ten full-attention layers with grouped-query attention, sixteen query
  heads and two key/value heads, into its stack: "Perplexity libera Lily: inferencia en Rust y
  Metal para Mac" (mechatronicstore.cl), section "Tres formas de carga en un mismo modelo";
  "Perplexity ouvre le code de Lily..." (lefilia.fr), article body.
* At decode the attention reads a key/value cache that grows with the context; the engine packs
  query heads of one group so that every key and value row is loaded once, and lays long
  contexts out in fixed blocks: same page, section "Decode: mover menos bytes por token".
Readings (the pages are silent): head size 128 (hidden size / query heads); query head h uses
key/value head h // (Hq / Hkv); scores are q . k / sqrt(head size); softmax over all cached
positions (the new token's key and value are already in the cache); bf16 query and cache, the
output in float64 here.
"""
from __future__ import annotations

import math

import numpy as np


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def gqa_decode_attention(q_bits, k_bits, v_bits) -> np.ndarray:
    """One decode step of grouped-query attention.

    q_bits  bf16 [Hq, D]         the new token's query heads
    k_bits  bf16 [Hkv, N, D]     key cache of the N cached positions
    v_bits  bf16 [Hkv, N, D]     value cache
    Returns o float64 [Hq, D]:  o_h = sum_n softmax_n(q_h . k_{g,n} / sqrt(D)) v_{g,n},
    g = h // (Hq / Hkv).  Grouped-query attention with sixteen query and two key/value heads:
    "Perplexity libera Lily..." (mechatronicstore.cl), section "Tres formas de carga en un mismo
    modelo"; the scaling and the head-to-group map are readings."""
    q = bf16_to_f64(q_bits)
    k = bf16_to_f64(k_bits)
    v = bf16_to_f64(v_bits)
    Hq, D = q.shape
    Hkv, N, _ = k.shape
    assert Hq % Hkv == 0 and N >= 1
    group = Hq // Hkv
    o = np.zeros((Hq, D))
    for h in range(Hq):
        g = h // group
        s = k[g] @ q[h] / math.sqrt(D)
        p = np.exp(s - s.max())
        o[h] = (p / p.sum()) @ v[g]
    return o


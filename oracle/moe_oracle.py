"""CPU oracle for the 4-bit mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, fp64 statement of what the
layer computes.  Only the test suite, the package smoke check and the CPU-baseline leg
of the benchmark may import it; the CUDA library and its Python binding never do, and
they share no code with it (the seeded input generators in `synth` are the only common
dependency, and they hold none of the layer's arithmetic).

What the layer computes, and where the pages say so (pages describing Perplexity's Lily
engine; quoted by site, page title and section):

* Weight format -- "Perplexity libera Lily: inferencia en Rust y Metal para Mac"
  (mechatronicstore.cl), section "Prefill: pesos comprimidos y enrutamiento en la GPU":
  4-bit affine quantisation by groups, every group of 64 weights shares one bf16 scale and
  one bf16 bias, so w = q * scale + bias.  The packing (eight codes per uint32, lowest
  nibble = lowest column, groups along the input dimension) is a reading; the pages do not
  state it.
* Router -- "Perplexity ouvre le code de Lily..." (lefilia.fr), article body, and the
  mechatronicstore.cl page, section "Tres formas de carga en un mismo modelo": a router
  scores 256 experts and keeps eight, plus one shared expert that every token uses.
  Top-k in descending logit order with ties to the lower expert index, and weights that
  are the softmax of the k selected logits, are readings (the pages name no function).
* Routing tables -- mechatronicstore.cl, section "Prefill...": a routing histogram, a
  prefix scan, a scatter and a block map are built on the GPU.  Their exact contents
  (counts, exclusive offsets, permutation sorted by (expert, token), tiles of at most
  tile_n rows per expert in (expert, tile) order, then the shared expert as group E) are
  readings; the pages name the tables, not their layout.
* Expert FFN -- the pages do not name the activation; SwiGLU h = silu(x Wg^T) * (x Wu^T),
  y = h Wd^T is the reading.  The pages state FP32 accumulation for the GPU GEMM; the oracle
  accumulates in fp64 (the exact reference), with an optional mode that rounds the GEMM
  operands (dequantised weights, x, h) to the 16-bit operand type of the tensor-core path.
* Shared expert gate -- sigmoid(x . w_sg) (reading; the pages name no gate).
* Combine -- y[t] = sum_j w[t,j] * Y_{e_j}(x_t) + sigmoid(x_t . w_sg) * Y_shared(x_t), in j order.
"""
from __future__ import annotations

import math

import numpy as np

GROUP = 64


# ------------------------------------------------------------------------------------------
# Number formats
# ------------------------------------------------------------------------------------------

def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_format(v, mant_bits: int, emin: int, emax: int) -> np.ndarray:
    """Round float64 values to a binary format with `mant_bits` significant bits
    (implicit bit included), minimum normal exponent `emin` and maximum exponent `emax`,
    round-to-nearest-even, with gradual underflow and overflow to +-inf.

    fp16: (11, -14, 15); bf16: (8, -126, 127).
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v, copy=True)
    finite = np.isfinite(v) & (v != 0)
    _, ex = np.frexp(v[finite])          # v = m * 2**ex with 0.5 <= |m| < 1
    e_unb = ex - 1                        # v = 1.xxx * 2**e_unb
    q_exp = np.maximum(e_unb, emin) - (mant_bits - 1)
    quantum = np.ldexp(1.0, q_exp)
    r = np.round(v[finite] / quantum) * quantum   # np.round: half to even; the division is exact
    maxval = (2.0 - 2.0 ** (1 - mant_bits)) * 2.0 ** emax
    r = np.where(np.abs(r) > maxval, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def round_fp16(v):
    return round_to_format(v, 11, -14, 15)


def round_bf16(v):
    return round_to_format(v, 8, -126, 127)


def round_fp32(v):
    return round_to_format(v, 24, -126, 127)


# ------------------------------------------------------------------------------------------
# 4-bit affine group-64 weights
# ------------------------------------------------------------------------------------------

def unpack_codes(codes) -> np.ndarray:
    """uint32 words [..., C/8] -> 4-bit codes [..., C]; column c = 8*w + i sits in bits 4i..4i+3.
    4-bit codes: "Perplexity libera Lily..." (mechatronicstore.cl),
    section "Prefill: pesos comprimidos y enrutamiento en la GPU"; the packing order is a
    reading (the pages do not give it)."""
    codes = np.asarray(codes, dtype=np.uint32)
    shifts = (4 * np.arange(8, dtype=np.uint32))
    q = (codes[..., None] >> shifts) & np.uint32(0xF)
    return q.reshape(codes.shape[:-1] + (codes.shape[-1] * 8,)).astype(np.uint8)


def dequant(codes, scales, biases) -> np.ndarray:
    """w[r, c] = q[r, c] * scale[r, c // 64] + bias[r, c // 64], exact in float64.
    Affine groups of 64 with one bf16 scale and one bf16 bias: "Perplexity libera Lily..."
    (mechatronicstore.cl), section "Prefill: pesos comprimidos y enrutamiento en la GPU"."""
    q = unpack_codes(codes).astype(np.float64)
    s = np.repeat(bf16_to_f64(scales), GROUP, axis=-1)
    b = np.repeat(bf16_to_f64(biases), GROUP, axis=-1)
    assert q.shape == s.shape == b.shape
    return q * s + b


def expert_weights(experts: dict, e: int) -> tuple:
    """Dequantised (Wg [F,d], Wu [F,d], Wd [d,F]) of expert e of a stacked expert set."""
    out = []
    for name in ("gate", "up", "down"):
        m = experts[name]
        out.append(dequant(m["codes"][e], m["scales"][e], m["biases"][e]))
    return tuple(out)


# ------------------------------------------------------------------------------------------
# Routing
# ------------------------------------------------------------------------------------------

def route_topk(logits, k: int):
    """Per token, the k largest fp32 logits in descending order; equal logits go to the lower
    expert index (-0.0 equals +0.0); NaN ranks below every number.  Weights are the softmax
    of the selected logits (renormalised over the k), computed in float64.
    A router keeps 8 of 256 experts: "Perplexity ouvre le code de Lily..." (lefilia.fr),
    article body, and "Perplexity libera Lily..." (mechatronicstore.cl), section "Tres formas
    de carga en un mismo modelo"; the order, the tie rule and the weight function are readings.

    Returns idx int32 [T,k] and w float64 [T,k].
    """
    lg = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = lg.shape
    assert 1 <= k <= E
    order = np.argsort(-lg, axis=1, kind="stable")   # stable: ties keep ascending index; NaN last
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(lg, idx.astype(np.int64), axis=1)
    ex = np.exp(sel - sel[:, :1])
    w = ex / ex.sum(axis=1, keepdims=True)
    return idx, w


def routing_tables(idx, E: int, tile_n: int, with_shared: bool = True) -> dict:
    """Histogram, exclusive scan, permutation and block map of the top-k assignments.
    The pages name these four steps ("Perplexity libera Lily..." (mechatronicstore.cl), section
    "Prefill: pesos comprimidos y enrutamiento en la GPU"); their layout below is a reading.

    Assignment a = t*k + j routes token t to expert idx[t, j].
      counts[e]   number of assignments to expert e                       int32 [E]
      offsets[e]  exclusive prefix sum of counts; offsets[E] = T*k          int32 [E+1]
      perm[p]     assignment in slot p; slots sorted by (expert, token)     int32 [T*k]
      inv[a]      slot of assignment a (inv[perm[p]] = p)                   int32 [T*k]
      tiles       [num_tiles, 3] rows (e, first slot, rows): for each non-empty expert in
                  increasing e, ceil(counts[e]/tile_n) tiles of at most tile_n slots; then, when
                  the layer has a shared expert, group E over slots T*k .. T*k+T-1 in token order.
    """
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int64)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    a = np.arange(T * k, dtype=np.int64)
    t_of_a = a // k
    e_of_a = idx.ravel()
    perm = a[np.lexsort((t_of_a, e_of_a))]          # primary key expert, then token
    inv = np.empty_like(perm)
    inv[perm] = np.arange(T * k)
    tiles = []
    for e in range(E):
        c = int(counts[e])
        for i in range(0, c, tile_n):
            tiles.append((e, int(offsets[e]) + i, min(tile_n, c - i)))
    if with_shared:
        for i in range(0, T, tile_n):
            tiles.append((E, T * k + i, min(tile_n, T - i)))
    return {
        "counts": counts.astype(np.int32),
        "offsets": offsets.astype(np.int32),
        "perm": perm.astype(np.int32),
        "inv": inv.astype(np.int32),
        "tiles": np.array(tiles, dtype=np.int32).reshape(-1, 3),
        "num_tiles": len(tiles),
    }


# ------------------------------------------------------------------------------------------
# Expert FFN, shared gate, layer
# ------------------------------------------------------------------------------------------

def silu(a):
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def sigmoid(a):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-a))


_ROUNDERS = {None: None, "fp16": round_fp16, "bf16": round_bf16}


def expert_ffn(xe, Wg, Wu, Wd, operands=None, out16=False):
    """SwiGLU expert: h = silu(xe Wg^T) * (xe Wu^T); returns h Wd^T.  float64 accumulation.

    operands: None for the exact path, or "fp16"/"bf16" to round the GEMM operands
    (weights, activations and h) to that type first, as the tensor-core path does.
    out16: also round the expert's output rows to a 16-bit type before the weighted combine, as
    the layer path of the tensor-core kernels stores them: True or "fp16" for fp16, "bf16" for
    bf16 (an emulation choice only: the pages fix no intermediate precision; the exact oracle
    never rounds).
    """
    rnd = _ROUNDERS[operands]
    if rnd is not None:
        Wg, Wu, Wd, xe = rnd(Wg), rnd(Wu), rnd(Wd), rnd(xe)
    g = xe @ Wg.T
    u = xe @ Wu.T
    h = silu(g) * u
    if rnd is not None:
        h = rnd(h)
    out = h @ Wd.T
    if not out16:
        return out
    return round_bf16(out) if out16 == "bf16" else round_fp16(out)


def shared_gate(x, w_sg_bits):
    """sigmoid(x . w_sg) per token (float64).  The always-on shared expert: "Perplexity libera
    Lily..." (mechatronicstore.cl), section "Tres formas de carga en un mismo modelo"; its
    sigmoid gate is a reading."""
    return sigmoid(np.asarray(x, dtype=np.float64) @ bf16_to_f64(w_sg_bits))


def moe_layer(x_bits, logits, layer: dict, k: int, tile_n: int = 128, operands=None, out16=False) -> dict:
    """One MoE layer: route, run every expert on its tokens (grouped by the permutation),
    run the shared expert on all tokens, and combine.  Returns y (float64 [T,d]) and the
    routing tables.  Composition of the steps above: "Perplexity libera Lily..." (mechatronicstore.cl),
    sections "Tres formas de carga en un mismo modelo" and "Prefill: pesos comprimidos y
    enrutamiento en la GPU"."""
    x = bf16_to_f64(x_bits)
    T, d = x.shape
    routed = layer["routed"]
    E = routed["gate"]["codes"].shape[0]
    idx, w = route_topk(logits, k)
    tab = routing_tables(idx, E, tile_n, with_shared=layer.get("shared") is not None)
    perm, inv, off = tab["perm"], tab["inv"], tab["offsets"]
    n_slots = T * k + (T if layer.get("shared") is not None else 0)
    Y = np.zeros((n_slots, d), dtype=np.float64)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        tokens = perm[lo:hi] // k
        Y[lo:hi] = expert_ffn(x[tokens], *expert_weights(routed, e), operands=operands, out16=out16)
    y = np.zeros((T, d), dtype=np.float64)
    for j in range(k):
        y += w[:, j:j + 1] * Y[inv[np.arange(T) * k + j]]
    gs = None
    if layer.get("shared") is not None:
        Y[T * k:] = expert_ffn(x, *expert_weights(layer["shared"], 0), operands=operands, out16=out16)
        gs = shared_gate(x, layer["w_sg"])
        y += gs[:, None] * Y[T * k:]
    out = dict(tab)
    out.update({"y": y, "idx": idx, "w": w, "Y_perm": Y, "gs": gs})
    return out


def moe_token(x_bits_row, logits_row, layer: dict, k: int, operands=None, out16=False):
    """The layer for one token (float64 [d]); the same definition, without routing tables.
    Used to check sampled tokens of large workloads one by one (same sources as moe_layer)."""
    x = bf16_to_f64(np.asarray(x_bits_row)[None, :])
    idx, w = route_topk(np.asarray(logits_row, dtype=np.float32)[None, :], k)
    y = np.zeros(x.shape[1], dtype=np.float64)
    for j in range(k):
        e = int(idx[0, j])
        y += w[0, j] * expert_ffn(x, *expert_weights(layer["routed"], e), operands=operands, out16=out16)[0]
    if layer.get("shared") is not None:
        gs = shared_gate(x, layer["w_sg"])[0]
        y += gs * expert_ffn(x, *expert_weights(layer["shared"], 0), operands=operands, out16=out16)[0]
    return y, idx[0], w[0]


# ------------------------------------------------------------------------------------------
# Pre-norm block for the layer stack: RMSNorm -> router -> MoE -> residual
# ------------------------------------------------------------------------------------------

def rmsnorm_bf16(x_resid, gamma_bits, eps: float):
    """h = x / sqrt(mean(x^2) + eps) * gamma, rounded to bf16 (the layer's input type).
    Returns (h float64 values, h bf16 bits).  The pre-norm block of the layer stack is a
    reading (the pages describe the MoE layer, not the blocks around it)."""
    x = np.asarray(x_resid, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    h = round_bf16(x * r * bf16_to_f64(gamma_bits))
    bits = (h.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    return h, bits


def router_logits(h, w_router_bits):
    """logits = h W_r^T, accumulated in float64 and rounded to fp32 (the routing input type).
    The router that scores the 256 experts: "Perplexity libera Lily..." (mechatronicstore.cl), section
    "Tres formas de carga en un mismo modelo"; a linear router is a reading."""
    return round_fp32(np.asarray(h, dtype=np.float64) @ bf16_to_f64(w_router_bits).T).astype(np.float32)


def stack_tokens(x0_rows, layers: list, routers: list, k: int, eps: float = 1e-6, operands=None,
                 forced_logits: list | None = None, out16=False):
    """The residual stack for a few independent tokens: for each layer,
    h = RMSNorm(x)*gamma (bf16), logits = h W_r^T, x <- x + MoE(h).  Tokens are independent,
    so any subset of rows can be checked alone.  `forced_logits[l]` (optional, [n, E]) replaces
    the oracle's own router logits of layer l (teacher forcing of the expert choice).
    Returns x (float64 [n, d]) and per-layer top-k indices."""
    x = np.asarray(x0_rows, dtype=np.float64).copy()
    picks = []
    for li, (layer, rt) in enumerate(zip(layers, routers)):
        h, hbits = rmsnorm_bf16(x, rt["gamma"], eps)
        lg = router_logits(h, rt["w_router"]) if forced_logits is None else forced_logits[li]
        ys, ids = [], []
        for i in range(x.shape[0]):
            y, idx, _ = moe_token(hbits[i], lg[i], layer, k, operands=operands, out16=out16)
            ys.append(y)
            ids.append(idx)
        x = x + np.stack(ys)
        picks.append(np.stack(ids))
    return x, picks

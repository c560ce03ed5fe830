"""Seeded synthetic inputs for the 4-bit MoE layer and the grouped-query decode attention (shared by
the tests, the oracle checks and bench.py).

This module only draws random numbers with the shapes and distributions of the
workloads; it holds none of the layer's arithmetic (no dequantisation, routing,
FFN or combine).  Both the CPU oracle and the CUDA path consume what it returns.

Weight format (one "qmat" of R output rows and C input columns):
  codes  uint32 [R, C/8]   eight 4-bit codes per word, column c in bits 4*(c%8)..4*(c%8)+3
  scales uint16 [R, C/64]  bf16 bit patterns, one per group of 64 input columns
  biases uint16 [R, C/64]  bf16 bit patterns
Routed experts stack a leading expert axis E; the shared expert uses a leading axis of 1.

Distributions (per workload table): codes uniform over 0..15 (a uniform uint32 word
is eight independent uniform nibbles), scale ~ U(0.005, 0.02) rounded to bf16,
bias = -8 * scale * (1 + U(-0.05, 0.05)) rounded to bf16, x ~ N(0,1) rounded to bf16,
router logits fp32 N(0,1) with a per-workload offset, shared-gate vector
w_sg ~ N(0,1)/sqrt(d) rounded to bf16.

Decode attention (16 query heads, 2 key/value heads, head size 128; contexts of 32K, 64K and
128K positions as in the pages' measurements): the query q ~ N(0, q_scale^2) and the cached keys
and values ~ N(0,1), all rounded to bf16, so the scaled scores q.k/sqrt(128) have standard
deviation q_scale; a cache allocated beyond the context holds a given fill pattern there.

Gated DeltaNet scan (16 heads, key and value size 128): q, k, v ~ N(0,1) rounded to bf16; the decay
a = exp(g) ~ U(0.90, 0.999) per token and head (g = log a in fp32); the write strength
b = sigmoid(z), z ~ N(0,1), in fp32; the initial state ~ N(0, 0.1^2) in fp32 (zero for a fresh
prompt).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GROUP = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    F: int
    F_shared: int
    logits: str = "normal"      # "normal" | "normal_jitter" | "zipf"
    layers: int = 1
    seed: int = 0


# The five workloads of the MoE layer, named by what they are.
TINY = Workload("tiny_T16_d256_E16_k2_F128", T=16, d=256, E=16, k=2, F=128, F_shared=128,
                logits="normal_jitter")
DECODE = Workload("decode_T1_d2048_E256_k8_F512", T=1, d=2048, E=256, k=8, F=512, F_shared=512)
PREFILL = Workload("prefill_T512_d2048_E256_k8_F512", T=512, d=2048, E=256, k=8, F=512, F_shared=512)
SKEWED = Workload("skewed_prefill_T4096_zipf1.1_d2048_E256_k8_F512", T=4096, d=2048, E=256, k=8,
                  F=512, F_shared=512, logits="zipf")
STACK = Workload("stack40_T2048_d2048_E256_k8_F512", T=2048, d=2048, E=256, k=8, F=512, F_shared=512,
                 layers=40)

WORKLOADS = {w.name: w for w in (TINY, DECODE, PREFILL, SKEWED, STACK)}


@dataclasses.dataclass(frozen=True)
class AttnWorkload:
    name: str
    Hq: int
    Hkv: int
    D: int
    N: int
    layers: int = 1


# Decode attention of the model's ten full-attention layers at the pages' context lengths.
GQA_SMALL = AttnWorkload("gqa_Hq16_Hkv2_D128_N4097", 16, 2, 128, 4097)
GQA_32K = AttnWorkload("gqa_decode10_Hq16_Hkv2_D128_N32768", 16, 2, 128, 32768, layers=10)
GQA_64K = AttnWorkload("gqa_decode10_Hq16_Hkv2_D128_N65536", 16, 2, 128, 65536, layers=10)
GQA_128K = AttnWorkload("gqa_decode10_Hq16_Hkv2_D128_N131072", 16, 2, 128, 131072, layers=10)


@dataclasses.dataclass(frozen=True)
class ScanWorkload:
    name: str
    T: int
    H: int
    D: int
    layers: int = 1
    fresh: bool = False   # zero initial state (a new prompt)


# The model's thirty Gated DeltaNet layers: a decode token, and prompts of 512 and 2048 tokens.
SCAN_DECODE = ScanWorkload("deltanet30_decode_T1_H16_D128", 1, 16, 128, layers=30)
SCAN_512 = ScanWorkload("deltanet_prefill_T512_H16_D128", 512, 16, 128, fresh=True)
SCAN_2048 = ScanWorkload("deltanet_prefill_T2048_H16_D128", 2048, 16, 128, fresh=True)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even) and return the 16-bit patterns."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def make_qmat(rng: np.random.Generator, lead: int, R: int, C: int) -> dict:
    assert C % GROUP == 0
    codes = rng.integers(0, 2**32, size=(lead, R, C // 8), dtype=np.uint32)
    g = C // GROUP
    scale = f32_to_bf16_bits(rng.uniform(0.005, 0.02, size=(lead, R, g)).astype(np.float32))
    jitter = rng.uniform(-0.05, 0.05, size=(lead, R, g)).astype(np.float32)
    bias = f32_to_bf16_bits(np.float32(-8.0) * bf16_bits_to_f32(scale) * (np.float32(1.0) + jitter))
    return {"codes": codes, "scales": scale, "biases": bias}


def make_experts(rng: np.random.Generator, lead: int, d: int, F: int) -> dict:
    """gate [lead,F,d], up [lead,F,d], down [lead,d,F] in the qmat format."""
    return {"gate": make_qmat(rng, lead, F, d), "up": make_qmat(rng, lead, F, d),
            "down": make_qmat(rng, lead, d, F)}


def make_layer(w: Workload, seed: int | None = None) -> dict:
    """Weights of one MoE layer: routed experts, shared expert and shared-gate vector."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    routed = make_experts(rng, w.E, w.d, w.F)
    shared = make_experts(rng, 1, w.d, w.F_shared) if w.F_shared > 0 else None
    w_sg = f32_to_bf16_bits((rng.standard_normal(w.d) / math.sqrt(w.d)).astype(np.float32))
    return {"routed": routed, "shared": shared, "w_sg": w_sg}


def zipf_logit_bias(E: int, s: float = 1.1) -> np.ndarray:
    """log p_e with p_e proportional to (e+1)^-s over E experts (rank = index + 1)."""
    p = (np.arange(1, E + 1, dtype=np.float64)) ** (-s)
    p /= p.sum()
    return np.log(p)


def make_logits(rng: np.random.Generator, w: Workload, T: int | None = None) -> np.ndarray:
    T = w.T if T is None else T
    base = rng.standard_normal((T, w.E))
    if w.logits == "normal_jitter":
        base = base + 1e-4 * np.arange(w.E)[None, :]
    elif w.logits == "zipf":
        base = base + zipf_logit_bias(w.E)[None, :]
    return base.astype(np.float32)


def make_x(rng: np.random.Generator, T: int, d: int) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((T, d)).astype(np.float32))


def make_inputs(w: Workload, seed: int | None = None, T: int | None = None) -> dict:
    """Token activations x (bf16 bits [T,d]) and router logits (fp32 [T,E])."""
    rng = np.random.default_rng((w.seed if seed is None else seed) + 1_000_003)
    T = w.T if T is None else T
    x = make_x(rng, T, w.d)
    logits = make_logits(rng, w, T)
    return {"x": x, "logits": logits}


def make_router(w: Workload, seed: int) -> dict:
    """Pre-norm block extras for the layer stack: RMSNorm weight gamma = 1 and router W_r ~ N(0,1)/sqrt(d)."""
    rng = np.random.default_rng(seed + 2_000_003)
    gamma = f32_to_bf16_bits(np.ones(w.d, dtype=np.float32))
    w_router = f32_to_bf16_bits((rng.standard_normal((w.E, w.d)) / math.sqrt(w.d)).astype(np.float32))
    return {"gamma": gamma, "w_router": w_router}


def make_attention(Hq: int, Hkv: int, D: int, N: int, capacity: int | None = None, seed: int = 0,
                   q_scale: float = 1.0, tail_bits: int | None = None) -> dict:
    """q bf16 [Hq, D]; k, v bf16 [Hkv, capacity, D] (bit patterns); positions >= N hold tail_bits
    when given."""
    rng = np.random.default_rng(seed + 3_000_017)
    cap = N if capacity is None else capacity
    q = f32_to_bf16_bits((rng.standard_normal((Hq, D)) * q_scale).astype(np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((Hkv, cap, D), dtype=np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((Hkv, cap, D), dtype=np.float32))
    if tail_bits is not None and cap > N:
        k[:, N:] = tail_bits
        v[:, N:] = tail_bits
    return {"q": q, "k": k, "v": v}


def make_scan(T: int, H: int, D: int, seed: int = 0, fresh: bool = False) -> dict:
    """q, k, v bf16 [T, H, D] (bit patterns); g, beta fp32 [T, H]; S0 fp32 [H, D, D]."""
    rng = np.random.default_rng(seed + 4_000_037)
    q = f32_to_bf16_bits(rng.standard_normal((T, H, D), dtype=np.float32))
    k = f32_to_bf16_bits(rng.standard_normal((T, H, D), dtype=np.float32))
    v = f32_to_bf16_bits(rng.standard_normal((T, H, D), dtype=np.float32))
    g = np.log(rng.uniform(0.90, 0.999, (T, H))).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))).astype(np.float32)
    S0 = np.zeros((H, D, D), np.float32) if fresh else (rng.standard_normal((H, D, D)) * 0.1).astype(np.float32)
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "S0": S0}


# ----------------------------------------------------------------------------------------------
# Device-side generation for the large benchmark workloads (same distributions, torch RNG stream).
# ----------------------------------------------------------------------------------------------

def torch_make_layer(w: Workload, seed: int, device) -> dict:
    """Same recipe as make_layer, drawn with torch's generator directly on `device`.

    The random stream differs from the numpy one; the shapes and distributions are identical.
    """
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def qmat(lead, R, C):
        codes = torch.randint(-2**31, 2**31, (lead, R, C // 8), generator=gen, device=device,
                              dtype=torch.int64).to(torch.int32)
        g = C // GROUP
        s = torch.empty((lead, R, g), device=device).uniform_(0.005, 0.02, generator=gen).to(torch.bfloat16)
        j = torch.empty((lead, R, g), device=device).uniform_(-0.05, 0.05, generator=gen)
        b = (-8.0 * s.float() * (1.0 + j)).to(torch.bfloat16)
        return {"codes": codes, "scales": s.view(torch.int16), "biases": b.view(torch.int16)}

    def experts(lead, F):
        return {"gate": qmat(lead, F, w.d), "up": qmat(lead, F, w.d), "down": qmat(lead, w.d, F)}

    routed = experts(w.E, w.F)
    shared = experts(1, w.F_shared) if w.F_shared > 0 else None
    w_sg = (torch.randn(w.d, generator=gen, device=device) / math.sqrt(w.d)).to(torch.bfloat16)
    return {"routed": routed, "shared": shared, "w_sg": w_sg.view(torch.int16)}


def torch_make_inputs(w: Workload, seed: int, device, T: int | None = None) -> dict:
    import torch

    T = w.T if T is None else T
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 1_000_003)
    x = torch.randn((T, w.d), generator=gen, device=device).to(torch.bfloat16)
    logits = torch.randn((T, w.E), generator=gen, device=device)
    if w.logits == "normal_jitter":
        logits = logits + 1e-4 * torch.arange(w.E, device=device, dtype=torch.float32)[None, :]
    elif w.logits == "zipf":
        logits = logits + torch.from_numpy(zipf_logit_bias(w.E)).to(device=device, dtype=torch.float32)[None, :]
    return {"x": x.view(torch.int16), "logits": logits.contiguous()}


def torch_make_attention(Hq: int, Hkv: int, D: int, N: int, seed: int, device, q_scale: float = 1.0) -> dict:
    """Same recipe as make_attention (capacity N), drawn with torch's generator on `device`."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 3_000_017)
    q = (torch.randn((Hq, D), generator=gen, device=device) * q_scale).to(torch.bfloat16)
    k = torch.randn((Hkv, N, D), generator=gen, device=device).to(torch.bfloat16)
    v = torch.randn((Hkv, N, D), generator=gen, device=device).to(torch.bfloat16)
    return {"q": q.view(torch.int16), "k": k.view(torch.int16), "v": v.view(torch.int16)}


def torch_make_scan(T: int, H: int, D: int, seed: int, device, fresh: bool = False) -> dict:
    """Same recipe as make_scan, drawn with torch's generator on `device`."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 4_000_037)
    bf = lambda shape: torch.randn(shape, generator=gen, device=device).to(torch.bfloat16).view(torch.int16)
    q, k, v = bf((T, H, D)), bf((T, H, D)), bf((T, H, D))
    g = torch.empty((T, H), device=device).uniform_(0.90, 0.999, generator=gen).log()
    beta = torch.sigmoid(torch.randn((T, H), generator=gen, device=device))
    S0 = torch.zeros((H, D, D), device=device) if fresh else torch.randn((H, D, D), generator=gen, device=device) * 0.1
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "S0": S0}

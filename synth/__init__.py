"""Seeded synthetic inputs for the 4-bit MoE layer (shared by the tests, the oracle checks and bench.py).

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

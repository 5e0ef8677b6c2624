"""Seeded synthetic inputs for the DoRA norm/compose workloads.

This module only draws random inputs; it holds none of the DoRA arithmetic.
The same arrays feed the CUDA library (through the binding) and the fp64
oracle used by the tests, so both sides always see identical bits.

Workloads (the shapes of the summary page "人工智能训练新突破：Anthropic团队破解
大模型微调内存瓶颈难题": its 8192-wide, rank-384 module with batch 3 x seq 5120,
its rank range 16..768, and attention / MLP projection shapes):

  tiny        out=in=512,   r=16,  T=256,   fp32 activations computed from x
  attn_proj   out=in=4096,  r=64,  T=8192,  bf16 activations (forward + norm)
  high_rank   out=in=8192,  r=384, T=15360, bf16 activations (full train step)
  rank_sweep  out=in=8192,  T=8192, r in {16,64,128,256,512,768}, bf16
  mlp_gate_up in=4096, out=14336, r=512, T=16384, bf16 (32 per stack)
  mlp_down    in=14336, out=4096, r=512, T=16384, bf16 (32 per stack)

Distributions (all seeded; seed = 1000*workload_index + module_index):
  W0 ~ N(0, 1/in), A ~ N(0, 1/in), B ~ N(0, sigma_B^2)
  m  = ||W0_i|| * (1 + N(0, sigma_m^2))      (g close to 1)
  s  = alpha / sqrt(r), alpha = 32              (rsLoRA scale)
  tiny:   x ~ N(0,1)[T,in]; base = x W0^T, lora = x A^T B^T (fp64, stored fp32)
  others: base ~ N(0,1), lora ~ N(0, r*sigma_B^2) drawn directly (the variances
          of x W0^T and x A^T B^T for x ~ N(0,1)), rounded to bf16
  grad_out ~ N(0,1)
bf16 arrays are returned as uint16 bit patterns (round to nearest even).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

ALPHA = 32.0

WORKLOAD_INDEX = {
    "tiny": 0,
    "attn_proj": 1,
    "high_rank": 2,
    "rank_sweep": 3,
    "mlp_gate_up": 4,
    "mlp_down": 4,
}


@dataclasses.dataclass(frozen=True)
class ModuleShape:
    name: str
    out: int
    inp: int
    r: int
    T: int
    act: str            # "f32" or "bf16"
    sigma_B: float
    sigma_m: float
    train: bool         # backward included
    harness_acts: bool  # base/lora formed from x (tiny only)

    @property
    def s(self) -> float:
        return ALPHA / math.sqrt(self.r)

    @property
    def act_bytes(self) -> int:
        return 4 if self.act == "f32" else 2


_BASE = {
    "tiny": ModuleShape("tiny", 512, 512, 16, 256, "f32", 0.02, 1e-3, True, True),
    "attn_proj": ModuleShape("attn_proj", 4096, 4096, 64, 8192, "bf16", 0.01, 1e-2, False, False),
    "high_rank": ModuleShape("high_rank", 8192, 8192, 384, 15360, "bf16", 0.01, 1e-2, True, False),
    "rank_sweep": ModuleShape("rank_sweep", 8192, 8192, 384, 8192, "bf16", 0.01, 1e-2, True, False),
    "mlp_gate_up": ModuleShape("mlp_gate_up", 14336, 4096, 512, 16384, "bf16", 0.01, 1e-2, True, False),
    "mlp_down": ModuleShape("mlp_down", 4096, 14336, 512, 16384, "bf16", 0.01, 1e-2, True, False),
}

RANK_SWEEP = (16, 64, 128, 256, 512, 768)
MLP_REPEATS = 32


def shape(name: str, **overrides) -> ModuleShape:
    """The named workload's module shape, optionally with fields replaced
    (e.g. a smaller T or out for a test that keeps the same distributions)."""
    return dataclasses.replace(_BASE[name], **overrides)


def seed_for(name: str, module: int = 0) -> int:
    return 1000 * WORKLOAD_INDEX[name] + module


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    t = (u >> np.uint32(16)) & np.uint32(1)
    t += np.uint32(0x7FFF)
    t += u
    t >>= np.uint32(16)
    return t.astype(np.uint16)


def _normal(rng: np.random.Generator, shape, scale: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return a


def make_weights(sh: ModuleShape, seed: int) -> dict:
    """W0 [out,in], A [r,in], B [out,r], m [out] (all float32) and scale s."""
    rng = np.random.default_rng([seed, 0])
    W0 = _normal(rng, (sh.out, sh.inp), 1.0 / math.sqrt(sh.inp))
    A = _normal(rng, (sh.r, sh.inp), 1.0 / math.sqrt(sh.inp))
    B = _normal(rng, (sh.out, sh.r), sh.sigma_B)
    noise = rng.standard_normal(size=sh.out)
    # magnitude initialised at the base row norm, perturbed so that g ~ 1
    row = np.linalg.norm(W0.astype(np.float64), axis=1)
    m = (row * (1.0 + sh.sigma_m * noise)).astype(np.float32)
    return {"W0": W0, "A": A, "B": B, "m": m, "s": sh.s}


def stress_magnitude(row_norm: np.ndarray, seed: int) -> np.ndarray:
    """The g ~ 1 stress set's magnitude: m_i = row_norm_i * (1 + U(-2^-9, 2^-9))
    as float32.  With row_norm = ||W0_i|| this is the literal definition of the
    high-rank workload's stress subset; with row_norm = the adapted norm n_i
    (from the oracle), g - 1 = m/n - 1 lies in bf16's collapse region, where a
    naive bf16 compose rounds g to 1 and loses the base correction."""
    rng = np.random.default_rng([seed, 3])
    u = rng.uniform(-2.0 ** -9, 2.0 ** -9, size=np.shape(row_norm))
    return (np.asarray(row_norm, np.float64) * (1.0 + u)).astype(np.float32)


def make_activations(sh: ModuleShape, seed: int, weights: dict | None = None) -> dict:
    """base, lora, grad_out [T,out]: float32 arrays for act='f32', uint16
    bf16 bit patterns for act='bf16'."""
    rng = np.random.default_rng([seed, 1])
    if sh.harness_acts:
        if weights is None:
            weights = make_weights(sh, seed)
        x = rng.standard_normal(size=(sh.T, sh.inp)).astype(np.float64)
        W0 = weights["W0"].astype(np.float64)
        A = weights["A"].astype(np.float64)
        B = weights["B"].astype(np.float64)
        base = x @ W0.T
        lora = (x @ A.T) @ B.T
        base = base.astype(np.float32)
        lora = lora.astype(np.float32)
    else:
        base = _normal(rng, (sh.T, sh.out), 1.0)
        lora = _normal(rng, (sh.T, sh.out), math.sqrt(sh.r) * sh.sigma_B)
    dy = _normal(rng, (sh.T, sh.out), 1.0)
    if sh.act == "bf16":
        base = f32_to_bf16_bits(base)
        lora = f32_to_bf16_bits(lora)
        dy = f32_to_bf16_bits(dy)
    return {"base": base, "lora": lora, "dy": dy}


def make_layer(sh: ModuleShape, seed: int) -> dict:
    """Inputs of the compose folded into its adjacent products: x [T, in],
    W0 [out, in], xa [T, r] and base [T, out] as bf16 bit patterns; B [out, r]
    and g [out] float32; the scale s.  W0 and B are the module's seeded
    weights (W0 rounded to bf16); x ~ N(0,1); xa ~ N(0,1), the distribution of
    x A^T for these x and A, drawn directly; base ~ N(0,1); g = 1 + N(0, sigma_m^2)."""
    rng = np.random.default_rng([seed, 2])
    w = make_weights(sh, seed)
    x = f32_to_bf16_bits(_normal(rng, (sh.T, sh.inp), 1.0))
    xa = f32_to_bf16_bits(_normal(rng, (sh.T, sh.r), 1.0))
    base = f32_to_bf16_bits(_normal(rng, (sh.T, sh.out), 1.0))
    g = (1.0 + sh.sigma_m * rng.standard_normal(size=sh.out)).astype(np.float32)
    return {"x": x, "W0": f32_to_bf16_bits(w["W0"]), "xa": xa, "B": w["B"], "g": g, "base": base, "s": sh.s}


def make_module(sh: ModuleShape, seed: int) -> dict:
    w = make_weights(sh, seed)
    a = make_activations(sh, seed, w)
    w.update(a)
    return w

"""torch.library registration of the DoRA hot path (integration only).

Seven custom ops; each allocates its outputs (and the library's workspace)
with torch and calls the C entry points of the same names on the current CUDA
stream.  No arithmetic happens here:

  torch.ops.dora.norm_factored(W0, A, B, m, s) -> (norm, g)
  torch.ops.dora.row_sumsq(W0) -> n0sq                       (bf16 W0: ||W0_i||^2, once)
  torch.ops.dora.norm_factored_bf16(W0, A, B, m, n0sq, s) -> (norm, g)   (bf16 W0, A, B)
  torch.ops.dora.compose(base, lora, m, g, norm, s) -> y
  torch.ops.dora.compose_bwd(dy, base, lora, g, norm, s) -> (d_base, d_lora, d_mag)
  torch.ops.dora.norm_factored_bwd(W0, A, B, norm, g, d_mag, s) -> (dA, dB)   (through the norm)
  torch.ops.dora.module(base, lora, W0, A, B, m, s) -> (y, norm, g)           (norm not detached)

``compose`` is differentiable in base, lora and m.  It takes m beside g (the
norm op's output g = m / norm) so that autograd can deliver dL/dm: with the
row norm treated as a constant in the backward (the method's page,
"人工智能训练新突破：Anthropic团队破解大模型微调内存瓶颈难题", says nothing about a
gradient through the norm; this is the reading the library follows),
dL/dm_j = sum_t dy_tj (base_tj + s lora_tj) / norm_j, which is exactly the
library's d_mag, and dL/dbase = g dy, dL/dlora = s g dy are its d_base and
d_lora.  The backward is therefore one call of dora_compose_bwd.

``module`` is the variant with the norm NOT detached: differentiable in base,
lora, A, B and m.  Its backward is one dora_compose_bwd call followed, when A
or B needs a gradient, by one dora_norm_factored_bwd call on the d_mag it
returned (dL/dn = -g d_mag); its norm and g outputs are not differentiable.

Inputs must be contiguous, row-major and on one CUDA device (the C ABI's
layout); m, n0sq, norm and g are float32, the weights float32 (bfloat16 for
the _bf16 norm and row_sumsq), activations float32 or bfloat16.
"""
from __future__ import annotations

import torch
from torch import Tensor

from . import (dora_compose_bwd, dora_compose_bwd_workspace, dora_compose_fwd, dora_norm_factored,
               dora_norm_factored_bf16, dora_norm_factored_bf16_workspace, dora_norm_factored_bwd,
               dora_norm_factored_bwd_workspace, dora_norm_factored_workspace, dora_row_sumsq_bf16)

__all__ = ["norm_factored", "row_sumsq", "norm_factored_bf16", "compose", "compose_bwd", "norm_factored_bwd",
           "module", "dora_module"]


def _contig(name: str, *ts: Tensor) -> None:
    for t in ts:
        if not t.is_contiguous():
            raise ValueError(f"dora::{name}: inputs must be contiguous (row-major)")


@torch.library.custom_op("dora::norm_factored", mutates_args=(), device_types="cuda")
def norm_factored(W0: Tensor, A: Tensor, B: Tensor, m: Tensor, s: float) -> tuple[Tensor, Tensor]:
    """n_i = ||W0_i + s (B A)_i|| (factored: base + cross + Gram terms) and g = m / n."""
    _contig("norm_factored", W0, A, B, m)
    out, inp = W0.shape
    r = A.shape[0]
    norm = torch.empty(out, device=W0.device, dtype=torch.float32)
    g = torch.empty_like(norm)
    ws = torch.empty(max(dora_norm_factored_workspace(out, inp, r), 1), dtype=torch.uint8, device=W0.device)
    dora_norm_factored(W0, A, B, m, s, norm, g, ws)
    return norm, g


@norm_factored.register_fake
def _norm_factored_fake(W0, A, B, m, s):
    out = W0.shape[0]
    return W0.new_empty(out, dtype=torch.float32), W0.new_empty(out, dtype=torch.float32)


@torch.library.custom_op("dora::row_sumsq", mutates_args=(), device_types="cuda")
def row_sumsq(W0: Tensor) -> Tensor:
    """||W0_i||^2 of a bfloat16 W0 in fp32 (fixed summation order)."""
    _contig("row_sumsq", W0)
    n0sq = torch.empty(W0.shape[0], device=W0.device, dtype=torch.float32)
    dora_row_sumsq_bf16(W0, n0sq)
    return n0sq


@row_sumsq.register_fake
def _row_sumsq_fake(W0):
    return W0.new_empty(W0.shape[0], dtype=torch.float32)


@torch.library.custom_op("dora::norm_factored_bf16", mutates_args=(), device_types="cuda")
def norm_factored_bf16(W0: Tensor, A: Tensor, B: Tensor, m: Tensor, n0sq: Tensor, s: float) -> tuple[Tensor, Tensor]:
    """The factored norm for bfloat16 W0, A, B with ||W0_i||^2 given (n0sq)."""
    _contig("norm_factored_bf16", W0, A, B, m, n0sq)
    out, inp = W0.shape
    r = A.shape[0]
    norm = torch.empty(out, device=W0.device, dtype=torch.float32)
    g = torch.empty_like(norm)
    ws = torch.empty(max(dora_norm_factored_bf16_workspace(out, inp, r), 1), dtype=torch.uint8, device=W0.device)
    dora_norm_factored_bf16(W0, A, B, m, n0sq, s, norm, g, ws)
    return norm, g


@norm_factored_bf16.register_fake
def _norm_factored_bf16_fake(W0, A, B, m, n0sq, s):
    out = W0.shape[0]
    return W0.new_empty(out, dtype=torch.float32), W0.new_empty(out, dtype=torch.float32)


@torch.library.custom_op("dora::compose_bwd", mutates_args=(), device_types="cuda")
def compose_bwd(dy: Tensor, base: Tensor, lora: Tensor, g: Tensor, norm: Tensor,
                s: float) -> tuple[Tensor, Tensor, Tensor]:
    """d_base = g dy, d_lora = s g dy, d_mag = sum_t dy (base + s lora) / norm."""
    _contig("compose_bwd", dy, base, lora, g, norm)
    T, out = dy.shape
    d_base = torch.empty_like(dy)
    d_lora = torch.empty_like(dy)
    d_mag = torch.empty(out, device=dy.device, dtype=torch.float32)
    ws = torch.empty(max(dora_compose_bwd_workspace(T, out), 1), dtype=torch.uint8, device=dy.device)
    dora_compose_bwd(dy, base, lora, g, norm, s, d_base, d_lora, d_mag, ws)
    return d_base, d_lora, d_mag


@compose_bwd.register_fake
def _compose_bwd_fake(dy, base, lora, g, norm, s):
    return torch.empty_like(dy), torch.empty_like(dy), dy.new_empty(dy.shape[1], dtype=torch.float32)


@torch.library.custom_op("dora::compose", mutates_args=(), device_types="cuda")
def compose(base: Tensor, lora: Tensor, m: Tensor, g: Tensor, norm: Tensor, s: float) -> Tensor:
    """y = base + (g - 1) base + g s lora (fp32 inside, one rounding to the activation dtype)."""
    _contig("compose", base, lora, g)
    y = torch.empty_like(base)
    dora_compose_fwd(base, lora, g, s, y)
    return y


@compose.register_fake
def _compose_fake(base, lora, m, g, norm, s):
    return torch.empty_like(base)


def _compose_setup(ctx, inputs, output):
    base, lora, m, g, norm, s = inputs
    ctx.save_for_backward(base, lora, g, norm)
    ctx.s = s


def _compose_backward(ctx, dy):
    base, lora, g, norm = ctx.saved_tensors
    d_base, d_lora, d_mag = compose_bwd(dy.contiguous(), base, lora, g, norm, ctx.s)
    return d_base, d_lora, d_mag, None, None, None


compose.register_autograd(_compose_backward, setup_context=_compose_setup)


@torch.library.custom_op("dora::norm_factored_bwd", mutates_args=(), device_types="cuda")
def norm_factored_bwd(W0: Tensor, A: Tensor, B: Tensor, norm: Tensor, g: Tensor, d_mag: Tensor,
                      s: float) -> tuple[Tensor, Tensor]:
    """dA, dB through the row norm for dL/dn = -g d_mag (d_mag as compose_bwd returns it)."""
    _contig("norm_factored_bwd", W0, A, B, norm, g, d_mag)
    out, inp = W0.shape
    r = A.shape[0]
    dA = torch.empty(r, inp, device=W0.device, dtype=torch.float32)
    dB = torch.empty(out, r, device=W0.device, dtype=torch.float32)
    ws = torch.empty(max(dora_norm_factored_bwd_workspace(out, inp, r), 1), dtype=torch.uint8, device=W0.device)
    dora_norm_factored_bwd(W0, A, B, norm, g, d_mag, s, dA, dB, ws)
    return dA, dB


@norm_factored_bwd.register_fake
def _norm_factored_bwd_fake(W0, A, B, norm, g, d_mag, s):
    return torch.empty_like(A, dtype=torch.float32), torch.empty_like(B, dtype=torch.float32)


@torch.library.custom_op("dora::module", mutates_args=(), device_types="cuda")
def module(base: Tensor, lora: Tensor, W0: Tensor, A: Tensor, B: Tensor, m: Tensor,
           s: float) -> tuple[Tensor, Tensor, Tensor]:
    """y = g (base + s lora) with n and g from the factored norm; returns (y, norm, g)."""
    _contig("module", base, lora, W0, A, B, m)
    out, inp = W0.shape
    r = A.shape[0]
    norm = torch.empty(out, device=W0.device, dtype=torch.float32)
    g = torch.empty_like(norm)
    ws = torch.empty(max(dora_norm_factored_workspace(out, inp, r), 1), dtype=torch.uint8, device=W0.device)
    dora_norm_factored(W0, A, B, m, s, norm, g, ws)
    y = torch.empty_like(base)
    dora_compose_fwd(base, lora, g, s, y)
    return y, norm, g


@module.register_fake
def _module_fake(base, lora, W0, A, B, m, s):
    out = W0.shape[0]
    return torch.empty_like(base), W0.new_empty(out, dtype=torch.float32), W0.new_empty(out, dtype=torch.float32)


def _module_setup(ctx, inputs, output):
    base, lora, W0, A, B, m, s = inputs
    _, norm, g = output
    ctx.save_for_backward(base, lora, W0, A, B, norm, g)
    ctx.s = s
    ctx.mark_non_differentiable(norm, g)


def _module_backward(ctx, dy, d_norm_out, d_g_out):
    base, lora, W0, A, B, norm, g = ctx.saved_tensors
    d_base, d_lora, d_mag = compose_bwd(dy.contiguous(), base, lora, g, norm, ctx.s)
    dA = dB = None
    if ctx.needs_input_grad[3] or ctx.needs_input_grad[4]:
        dA, dB = norm_factored_bwd(W0, A, B, norm, g, d_mag, ctx.s)
    return d_base, d_lora, None, dA, dB, d_mag, None


module.register_autograd(_module_backward, setup_context=_module_setup)


def dora_module(base: Tensor, lora: Tensor, W0: Tensor, A: Tensor, B: Tensor, m: Tensor, s: float,
                detach_norm: bool = True) -> Tensor:
    """One DoRA module's output from its two matmul results.

    detach_norm=True (the page's backward): the factored norm carries no
    gradient; the fused compose is differentiable in base, lora and m.
    detach_norm=False: the gradient also flows through the norm into A and B
    (dora::module)."""
    if not detach_norm:
        return module(base, lora, W0.detach(), A, B, m, s)[0]
    norm, g = norm_factored(W0.detach(), A.detach(), B.detach(), m.detach(), s)
    return compose(base, lora, m, g, norm, s)

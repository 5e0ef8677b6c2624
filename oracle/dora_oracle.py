"""Plain fp64 CPU oracle for the DoRA weight-norm and compose path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` use it.  It shares no code with the CUDA library.

Source of the method (cited by paragraph below as "P1 ¶<opening words>"):
  P1 = web page "人工智能训练新突破：Anthropic团队破解大模型微调内存瓶颈难题"
       (techwalker.com, 2026-04-01), a summary of arXiv:2603.22276.

What it computes, written as the plain definitions (no blocking, no fusion,
no factoring -- the dense matrix W0 + s*B@A IS formed here on purpose, since
the whole point of the method is that the GPU path never forms it):

  * DoRA re-parametrisation (P1 ¶目前最流行的模型微调技术叫做DoRA, which names
    "weight-decomposed low-rank adaptation" and the per-module norm):
        W'   = m * (W0 + s B A) / ||W0 + s B A||_row
    with W0[out,in], A[r,in], B[out,r], magnitude m[out] and scale s.
    Row i of the adapted weight has norm n_i and magnitude scale g_i = m_i/n_i.
  * Layer output, for activations base = x W0^T and lora = x A^T B^T
    (lora is NOT pre-scaled; P1 ¶从技术架构角度来看 writes g*s*lora):
        y = g * (base + s * lora)                      (plain definition)
          = base + (g-1)*base + g*s*lora               (the page's stable form)
  * Backward with the norm treated as a constant (P1 is silent; reading c2):
        d_base = g*dy,  d_lora = s*g*dy,
        d_mag_j = sum_t dy[t,j]*(base[t,j] + s*lora[t,j]) / n_j .
  * The compose with its adjacent products folded in (compose_lora_fwd,
    linear_fwd): the same y, from xa = x A^T and the weights instead of from
    base and lora.
  * Variant with the norm NOT detached (gradient through n into A and B): the
    chain rule through g = m/n and n_i = ||V_i||, V = W0 + s B A (norm_grad).

Readings of silent or garbled points are listed in the repository design notes;
the ones that change arithmetic are repeated at the function that takes them.

bf16 handling: activations may arrive as bfloat16 bit patterns (uint16).  They
are widened exactly to fp64 here; the correctly rounded fp64 -> bf16 encoder
below is used to report the correctly rounded result of a computation.

Pins (tests/test_oracle.py): B = 0 against numpy.linalg.norm; Pythagoras and
parallel-row closed forms with orthonormal A; invariance of the norm under a
joint column permutation of W0 and A; the factored fp64 identity on
brute-force tiny shapes; hand-computed fixtures in tests/golden/; central
finite differences of L(m, base, lora) = <dy, y>; the homogeneity identity
sum_j m_j d_mag_j = sum dy*y; exact bf16 encodings against torch and against
hand-made double-rounding cases; for norm_grad, central finite differences
of L(A, B) = <w, g(A, B)>, torch autograd of the dense definition, Euler's
identity for the degree-1 homogeneous norm (W0 = 0) and the B = 0 closed form.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits_to_f64",
    "f64_to_bf16_bits",
    "adapted_row_norm",
    "weight_norm",
    "compose_fwd",
    "compose_fwd_stable",
    "compose_fwd_naive_bf16",
    "compose_bwd",
    "norm_grad",
    "compose_lora_fwd",
    "linear_fwd",
]


# ----------------------------------------------------------------------------
# bfloat16 <-> fp64 (exact widening; correctly rounded narrowing)
# ----------------------------------------------------------------------------

def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns (uint16) to fp64.

    A bfloat16 is the top half of an IEEE binary32, so shifting the 16 bits into
    the high half of a uint32 gives the identical binary32 value.
    """
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


_BF16_MIN_NORMAL = 2.0 ** -126
_BF16_SUBNORMAL_QUANTUM = 2.0 ** -133


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round fp64 values to bfloat16 with ONE round-to-nearest-even step.

    (Going through binary32 first would round twice and can differ.)
    Normal range: bfloat16 keeps 7 of fp64's 52 fraction bits, so the low 45
    bits are rounded away with ties to even; a carry into the exponent is the
    correct result.  Subnormal range (|x| < 2^-126): the grid is the fixed
    quantum 2^-133; numpy.rint rounds half to even.  Values past the largest
    finite bfloat16 become infinities through the binary32 cast.  NaN is not
    expected on this path and is not treated specially.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    small = np.abs(x) < _BF16_MIN_NORMAL
    # subnormal / zero: fixed-point grid
    out[small] = np.rint(x[small] / _BF16_SUBNORMAL_QUANTUM) * _BF16_SUBNORMAL_QUANTUM
    # normal: round the fp64 bit pattern at bit 45
    big = ~small
    bits = x[big].view(np.uint64)
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    bits = (bits + np.uint64((1 << 44) - 1) + lsb) & ~np.uint64((1 << 45) - 1)
    out[big] = bits.view(np.float64)
    # every value of `out` is now a bfloat16 value (or beyond range), so the
    # binary32 cast below is exact and the top 16 bits are the encoding
    with np.errstate(over="ignore"):
        f32 = out.astype(np.float32)
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


# ----------------------------------------------------------------------------
# (a) per-output-row weight norm and magnitude scale
# ----------------------------------------------------------------------------

def adapted_row_norm(W0, A, B, s) -> np.ndarray:
    """n_i = || W0_i + s (B A)_i ||_2 for every output row i, in fp64.

    P1 ¶第一个创新是"因式分解规范化"技术: the page splits this norm into a base,
    a cross and a Gram term so that the out x in matrix is never formed.  The
    oracle does the opposite on purpose: it forms the dense adapted weight and
    takes plain row norms, which is the quantity the factored form must equal.
    Norm axis: per output row of W0[out, in] (reading c1).
    Rows are independent, so passing a subset of rows of W0 and B gives the
    norms of exactly those rows.
    """
    W0 = _f64(W0)
    A = _f64(A)
    B = _f64(B)
    W = W0 + s * (B @ A)                 # dense adapted weight [out, in]
    return np.sqrt(np.sum(W * W, axis=1))


def weight_norm(W0, A, B, m, s):
    """Return (n, g) with n the adapted row norm and g = m / n (IEEE division).

    No epsilon is added (the page adds none; reading c5): n = 0 gives an
    infinite or NaN g exactly as IEEE division does.
    """
    n = adapted_row_norm(W0, A, B, s)
    with np.errstate(divide="ignore", invalid="ignore"):
        g = _f64(m) / n
    return n, g


# ----------------------------------------------------------------------------
# (b) compose forward / backward
# ----------------------------------------------------------------------------

def compose_fwd(base, lora, g, s) -> np.ndarray:
    """Plain DoRA layer output y = g * (base + s*lora), fp64.

    base, lora: [T, out]; g: [out] broadcast over tokens (rows).
    """
    base = _f64(base)
    lora = _f64(lora)
    g = _f64(g)
    return g[None, :] * (base + s * lora)


def compose_fwd_stable(base, lora, g, s) -> np.ndarray:
    """The page's stable form y = base + (g-1)*base + g*s*lora, fp64.

    P1 ¶从技术架构角度来看 gives this form: the small correction (g-1) is kept
    explicit so that it is not lost when g is close to 1.  In exact arithmetic
    it equals compose_fwd; in fp64 the two agree to rounding.
    """
    base = _f64(base)
    lora = _f64(lora)
    g = _f64(g)[None, :]
    return base + (g - 1.0) * base + g * s * lora


def compose_fwd_naive_bf16(base_bits, lora_bits, g, s) -> np.ndarray:
    """A naive bf16 evaluation of g*(base + s*lora), returned as bf16 bits.

    Used only to REPORT how much a naive low-precision compose loses near
    g = 1 (P1 ¶他们在一个Qwen2-VL-7B适配器上的测量: in the bf16 "collapse
    region" the base correction vanishes).  The page does not write the naive
    path out; the reading taken (c4) is four separate elementwise passes, each
    rounding its result to bf16, with g itself rounded to bf16:
        t1 = RN(s*lora);  t2 = RN(base + t1);  y = RN(RN(g) * t2).
    Each step is computed exactly in fp64 from bf16 operands (products and sums
    of two bf16 values are exact in fp64) and then rounded once.
    """
    b = bf16_bits_to_f64(base_bits)
    l = bf16_bits_to_f64(lora_bits)
    g16 = bf16_bits_to_f64(f64_to_bf16_bits(_f64(g)))[None, :]
    s16 = bf16_bits_to_f64(f64_to_bf16_bits(np.float64(s)))
    t1 = bf16_bits_to_f64(f64_to_bf16_bits(s16 * l))
    t2 = bf16_bits_to_f64(f64_to_bf16_bits(b + t1))
    return f64_to_bf16_bits(g16 * t2)


def compose_bwd(dy, base, lora, g, n, s):
    """Gradients of the compose with the row norm n held constant, fp64.

    y = (m/n) * (base + s*lora) with g = m/n, so
        d_base = g * dy
        d_lora = s * g * dy
        d_mag_j = (1/n_j) * sum_t dy[t,j] * (base[t,j] + s*lora[t,j]).
    P1 ¶研究团队在六个不同的GPU上 / ¶研究团队还进行了广泛的收敛等价性验证 name the
    fused backward and its d_mag output; the norm is detached (reading c2),
    so no gradient flows into A or B through n.
    Columns are independent, so passing a column subset (with the matching
    entries of g and n) gives exactly those columns.
    Returns (d_base [T,out], d_lora [T,out], d_mag [out]).
    """
    dy = _f64(dy)
    base = _f64(base)
    lora = _f64(lora)
    g = _f64(g)[None, :]
    n = _f64(n)
    d_base = g * dy
    d_lora = s * g * dy
    d_mag = np.sum(dy * (base + s * lora), axis=0) / n
    return d_base, d_lora, d_mag


# ----------------------------------------------------------------------------
# (c) the variant with the norm not detached: gradient through n into A, B
# ----------------------------------------------------------------------------

def norm_grad(W0, A, B, s, n, g, d_mag):
    """Gradients w.r.t. A and B that flow through the row norm, fp64.

    The page is silent on a gradient through the norm (its backward treats n
    as a constant; reading c2).  This is the other plain reading: n is a
    function of A and B.  The loss sees n only through g = m/n, and d_mag is
    dL/dm along that route (as compose_bwd returns it), i.e.
        dL/dg_i = d_mag_i * n_i,   dg_i/dn_i = -m_i/n_i^2 = -g_i/n_i
        =>  dL/dn_i = -g_i * d_mag_i .
    With V = W0 + s B A (dense) and dn_i/dV_i = V_i / n_i,
        dV  = (dL/dn / n)[:, None] * V
        dB  = s * dV @ A^T          (V = ... + s B A, so dV/dB carries s A)
        dA  = s * B^T @ dV .
    n and g are the forward's values, passed in (the backward of the library
    takes them as inputs too); V is formed densely from the weights.
    Rows are independent for dB (a row subset of W0, B, n, g, d_mag gives
    those rows of dB); columns are independent for dA (a column subset of W0
    and A, with all rows, gives those columns of dA).
    Returns (dA [r, in], dB [out, r]).
    """
    W0 = _f64(W0)
    A = _f64(A)
    B = _f64(B)
    n = _f64(n)
    dn = -_f64(g) * _f64(d_mag)
    V = W0 + s * (B @ A)
    dV = (dn / n)[:, None] * V
    return s * (B.T @ dV), s * (dV @ A.T)


# ----------------------------------------------------------------------------
# (d) the compose with its adjacent products: y from x, W0, xa = x A^T, B
# ----------------------------------------------------------------------------

def compose_lora_fwd(base, xa, B, g, s) -> np.ndarray:
    """y = g * (base + s * lora) with lora = xa B^T formed here, fp64.

    The layer's products on either side of the compose (P1 ¶从技术架构角度来看:
    base = x W0^T and lora = (x A^T) B^T); xa [T, r] is x A^T.  The matmul is
    numpy's in fp64; the compose is compose_fwd.
    """
    return compose_fwd(base, _f64(xa) @ _f64(B).T, g, s)


def linear_fwd(x, W0, xa, B, g, s) -> np.ndarray:
    """y = g * (x W0^T + s * xa B^T), the whole DoRA layer output, fp64."""
    return compose_fwd(_f64(x) @ _f64(W0).T, _f64(xa) @ _f64(B).T, g, s)

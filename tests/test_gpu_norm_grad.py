"""GPU parity of dora_norm_factored_bwd (gradient through the row norm into A
and B) against the fp64 oracle's norm_grad, through the C ABI.

Inputs: the seeded weights of the parity shapes; n and g from the oracle's
dense norm, rounded to fp32 (the backward's inputs -- both sides receive the
same fp32 values, so no input of the oracle comes from the library); d_mag
drawn from a seeded normal.

Tolerance, derived from the arithmetic.  Every output element is a sum of
products evaluated with the bf16 three-product split (x = h + l with h =
bf16(x), l = bf16(x - h); per product the dropped l l term and the residuals
are <= 3 * 2^-18 of its magnitude, see dora_norm_factored) and fp32
accumulation; dA also carries the error of s^2 H, itself such a sum.  (For
r <= 256, s G and s^2 H are fp32 FMA sums on the CUDA cores, whose error
lies within the same bound.)  With |.| the same expressions over absolute
values (abs_ref), a rigorous elementwise bound is
    |err| <= (2^-16 + 2^-23 (K + 64)) * abs_ref,   K = out + in + 2 r
(2^-23 per addition allows for an accumulator that truncates).  Because that
bound grows with K, the normwise error is also held to the norm's own
tolerance:  ||err||_F <= 1e-5 ||ref||_F.
"""
import numpy as np
import pytest
import torch

import oracle
from parameter_efficient_fine_gb300 import workloads as wl
import parameter_efficient_fine_gb300 as dora

from gpu_util import DEV, assert_no_device_error, f32_dev, run_norm, to_f64

pytestmark = pytest.mark.gpu

FRO_REL = 1e-5


def run_norm_bwd(W0, A, B, norm, g, d_mag, s):
    out, inp = W0.shape
    r = A.shape[0]
    dA = torch.full((r, inp), float("nan"), device=DEV)
    dB = torch.full((out, r), float("nan"), device=DEV)
    ws = torch.empty(max(dora.dora_norm_factored_bwd_workspace(out, inp, r), 1), dtype=torch.uint8, device=DEV)
    dora.dora_norm_factored_bwd(W0, A, B, norm, g, d_mag, s, dA, dB, ws)
    return dA, dB


def abs_refs(W0, A, B, s, n, g, d_mag):
    """Magnitude scales of dA and dB: the same sums over absolute values."""
    c = np.abs(g * d_mag / n)
    aY = s * c[:, None] * np.abs(B)                    # |s c B|, [out, r]
    aA, aW, aB = np.abs(A), np.abs(W0), np.abs(B)
    dA_abs = aY.T @ aW + (s * (aB.T @ aY)) @ aA        # |Y^T W0| + |s^2 H A|
    dB_abs = s * c[:, None] * (aW @ aA.T + s * aB @ (aA @ aA.T))
    return dA_abs, dB_abs


def check_grad(name, got, ref, absref, K):
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    bound = (2.0 ** -16 + 2.0 ** -23 * (K + 64)) * absref + 1e-30
    bad = int(np.count_nonzero(err > bound))
    assert bad == 0, f"{name}: {bad} elements over the bound (worst ratio {float(np.max(err / bound)):.3f})"
    fro = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300))
    assert fro <= FRO_REL, f"{name}: ||err||/||ref|| = {fro:.3e} > {FRO_REL:.0e}"
    return fro


def _case(out, inp, r, seed):
    sh = wl.shape("high_rank", out=out, inp=inp, r=r, T=1)
    d = wl.make_module(sh, seed)
    rng = np.random.default_rng(seed + 1)
    d_mag = (0.1 * rng.standard_normal(out)).astype(np.float32)
    return d, d_mag


def oracle_norm_f32(d, rows=None):
    """The oracle's n and g rounded to fp32 (inputs of the backward on both sides)."""
    W0, B, m = (d[k] if rows is None else d[k][rows] for k in ("W0", "B", "m"))
    n, g = oracle.weight_norm(W0, d["A"], B, m, d["s"])
    return n.astype(np.float32), g.astype(np.float32)


def _run_and_check(d, d_mag):
    s = d["s"]
    W0, A, B = (f32_dev(d[k]) for k in ("W0", "A", "B"))
    n32, g32 = oracle_norm_f32(d)
    norm, g = f32_dev(n32), f32_dev(g32)
    dm = f32_dev(d_mag)
    dA, dB = run_norm_bwd(W0, A, B, norm, g, dm, s)
    assert_no_device_error()
    n32, g32 = n32.astype(np.float64), g32.astype(np.float64)
    dA_ref, dB_ref = oracle.norm_grad(d["W0"], d["A"], d["B"], s, n32, g32, d_mag)
    dA_abs, dB_abs = abs_refs(d["W0"].astype(np.float64), d["A"].astype(np.float64), d["B"].astype(np.float64), s,
                              n32, g32, d_mag.astype(np.float64))
    out, inp = d["W0"].shape
    r = d["A"].shape[0]
    K = out + inp + 2 * r
    check_grad("dA", to_f64(dA), dA_ref, dA_abs, K)
    check_grad("dB", to_f64(dB), dB_ref, dB_abs, K)
    return dA, dB


@pytest.mark.parametrize("out,inp,r", [
    (512, 512, 16),       # the tiny workload's weight shape
    (1000, 1040, 384),    # ragged M tiles on both passes, N = 256 + 128 MMAs
    (300, 256, 1),        # r = 1, B padded to a 16-byte row
    (257, 512, 17),       # r not a multiple of 4 or 16
    (384, 256, 272),      # one N chunk of 272
    (200, 128, 400),      # two N chunks of 208
    (130, 64, 768),       # two N chunks of 384
    (8, 4, 5),            # one K block, mostly out of bounds
    (1, 16, 2),           # a single output row
    (300, 1040, 128),     # N = 128: 32-wide K blocks
    (260, 200, 129),      # N = 144
    (1030, 136, 64),      # out (the K of the dA pass) ragged against every K block width
    (200, 136, 32),       # CUDA-core Gram products: the largest r of 32 x 32 tiles
    (200, 136, 33),       # the smallest r of 64 x 64 tiles
    (2000, 4104, 256),    # the largest r of the CUDA-core Gram; slices longer than 128 (one wave)
    (300, 520, 257),      # the smallest r of the tensor-core Gram passes
    (400, 520, 100),      # N-side tile of 112 rows: one MMA over the stacked h and l rows (N = 224)
    (260, 200, 113),      # N-side tile of 128 rows, the largest so taken (N = 256)
])
def test_norm_grad_shapes(out, inp, r):
    d, d_mag = _case(out, inp, r, 9100 + out + r)
    _run_and_check(d, d_mag)


@pytest.mark.parametrize("k", range(10))
def test_norm_grad_drawn_shapes(k):
    # a seeded draw over the accepted shapes (in a multiple of 4, any r and out)
    rng = np.random.default_rng(20261205 + k)
    out, inp, r = int(rng.integers(1, 1300)), 4 * int(rng.integers(1, 326)), int(rng.integers(1, 801))
    d, d_mag = _case(out, inp, r, 9900 + k)
    _run_and_check(d, d_mag)


def test_norm_grad_is_bitwise_reproducible():
    d, d_mag = _case(1000, 1040, 384, 9201)
    s = d["s"]
    W0, A, B, m = (f32_dev(d[k]) for k in ("W0", "A", "B", "m"))
    norm, g = run_norm(W0, A, B, m, s)
    dm = f32_dev(d_mag)
    a1, b1 = run_norm_bwd(W0, A, B, norm, g, dm, s)
    a2, b2 = run_norm_bwd(W0, A, B, norm, g, dm, s)
    assert torch.equal(a1, a2) and torch.equal(b1, b2)


def test_zero_upstream_gives_zero_gradients():
    d, _ = _case(260, 200, 129, 9202)
    s = d["s"]
    W0, A, B, m = (f32_dev(d[k]) for k in ("W0", "A", "B", "m"))
    norm, g = run_norm(W0, A, B, m, s)
    dA, dB = run_norm_bwd(W0, A, B, norm, g, torch.zeros_like(norm), s)
    assert torch.count_nonzero(dA).item() == 0 and torch.count_nonzero(dB).item() == 0


def test_zero_b_gives_zero_da_and_closed_form_db():
    d, d_mag = _case(300, 1040, 128, 9203)
    d["B"] = np.zeros_like(d["B"])
    dA, dB = _run_and_check(d, d_mag)
    assert torch.count_nonzero(dA).item() == 0


def test_empty_rows_zero_da():
    inp, r = 64, 8
    A = torch.randn(r, inp, device=DEV)
    W0 = torch.empty(0, inp, device=DEV)
    B = torch.empty(0, r, device=DEV)
    e = torch.empty(0, device=DEV)
    dA, dB = run_norm_bwd(W0, A, B, e, e, e, 1.0)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dA).item() == 0 and dB.numel() == 0


@pytest.mark.parametrize("r", [16, 384, 768])
def test_full_size_sampled(r):
    # the high-rank module (out = in = 8192): dB on sampled rows, dA on sampled
    # columns, each from the oracle on exactly the rows / columns it needs
    sh = wl.shape("high_rank", r=r, T=1)
    d = wl.make_module(sh, wl.seed_for("high_rank") + r)
    s = d["s"]
    out, inp = d["W0"].shape
    rng = np.random.default_rng(9300 + r)
    d_mag = (0.1 * rng.standard_normal(out)).astype(np.float32)
    W0, A, B = (f32_dev(d[k]) for k in ("W0", "A", "B"))
    n32, g32 = oracle_norm_f32(d)
    dA, dB = run_norm_bwd(W0, A, B, f32_dev(n32), f32_dev(g32), f32_dev(d_mag), s)
    assert_no_device_error()
    n32, g32 = n32.astype(np.float64), g32.astype(np.float64)
    rows = np.sort(rng.choice(out, 96, replace=False))
    cols = np.sort(rng.choice(inp, 96, replace=False))
    rows[0], cols[-1] = 0, inp - 1
    _, dB_ref = oracle.norm_grad(d["W0"][rows], d["A"], d["B"][rows], s, n32[rows], g32[rows], d_mag[rows])
    dA_ref, _ = oracle.norm_grad(d["W0"][:, cols], d["A"][:, cols], d["B"], s, n32, g32, d_mag)
    W64, A64, B64 = (d[k].astype(np.float64) for k in ("W0", "A", "B"))
    dA_abs, _ = abs_refs(W64[:, cols], A64[:, cols], B64, s, n32, g32, d_mag.astype(np.float64))
    _, dB_abs = abs_refs(W64[rows], A64, B64[rows], s, n32[rows], g32[rows], d_mag[rows].astype(np.float64))
    K = out + inp + 2 * r
    check_grad("dA", to_f64(dA)[:, cols], dA_ref, dA_abs, K)
    check_grad("dB", to_f64(dB)[rows], dB_ref, dB_abs, K)

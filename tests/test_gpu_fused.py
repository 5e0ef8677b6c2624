"""GPU parity of the compose folded into its adjacent products
(dora_compose_lora_fwd, dora_compose_lora_fwd_bf16, dora_linear_fwd) against
the fp64 oracle, through the C ABI.  The bf16-B form gets B rounded to bf16,
and the oracle the same bf16 values.  Tolerance: the bf16 rule of tests/gpu_util.py (|err| <= 2^-7 |ref| +
1e-3 elementwise, cosine >= 0.99999).  The fraction of outputs equal to the
correctly rounded bf16 of the exact result is also checked: y is rounded once
from an fp32 accumulator whose error is far below half a bf16 ulp, so almost
every element is the correctly rounded one (a lost term or a wrong scale
drops this fraction to a few percent)."""
import numpy as np
import pytest
import torch

import oracle
import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import DEV, act_to_dev, assert_no_device_error, check_bf16_rule, f32_dev, to_f64

pytestmark = pytest.mark.gpu

CR_MIN = 0.95    # fraction of outputs that are the correctly rounded bf16 of the exact result


@pytest.fixture(params=["pairs", "single"])
def layout(request):
    """The fused kernel on CTA pairs (the default on GB300) or as single CTAs
    (the layout of a device without clusters of two, forced by the test hook)."""
    dora.dora_test_fused_pairs(request.param == "pairs")
    yield request.param
    dora.dora_test_fused_pairs(True)


def _layer(T, inp, out, r, seed):
    sh = wl.shape("high_rank", T=T, inp=inp, out=out, r=r)
    return wl.make_layer(sh, seed)


def _ws(out, r):
    return torch.empty(max(dora.dora_compose_fused_workspace(out, r), 1), dtype=torch.uint8, device=DEV)


def run_lora(d):
    base, xa = act_to_dev(d["base"]), act_to_dev(d["xa"])
    B, g = f32_dev(d["B"]), f32_dev(d["g"])
    y = torch.full_like(base, float("nan"))
    dora.dora_compose_lora_fwd(base, xa, B, g, d["s"], y, _ws(B.shape[0], B.shape[1]))
    return y


def run_lora_bf16(d):
    """The lora form for a bf16 B (B rounded to bf16 by the seeded generator's
    rounding; the oracle receives the same values)."""
    base, xa = act_to_dev(d["base"]), act_to_dev(d["xa"])
    Bb, g = act_to_dev(wl.f32_to_bf16_bits(d["B"])), f32_dev(d["g"])
    y = torch.full_like(base, float("nan"))
    dora.dora_compose_lora_fwd_bf16(base, xa, Bb, g, d["s"], y)
    return y


def ref_lora_bf16(d, rows=slice(None)):
    return oracle.compose_lora_fwd(_f64(d["base"][rows]), _f64(d["xa"][rows]), _f64(wl.f32_to_bf16_bits(d["B"])),
                                   d["g"], d["s"])


def run_linear(d):
    x, W0, xa = act_to_dev(d["x"]), act_to_dev(d["W0"]), act_to_dev(d["xa"])
    B, g = f32_dev(d["B"]), f32_dev(d["g"])
    y = torch.full((x.shape[0], W0.shape[0]), float("nan"), device=DEV, dtype=torch.bfloat16)
    dora.dora_linear_fwd(x, W0, xa, B, g, d["s"], y, _ws(B.shape[0], B.shape[1]))
    return y


def _check(name, y, ref):
    got = to_f64(y)
    assert np.all(np.isfinite(got)), f"{name}: non-finite outputs"
    check_bf16_rule(name, got, ref)
    cr = float(np.mean(got == oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(ref))))
    assert cr >= CR_MIN, f"{name}: only {cr:.4f} of outputs correctly rounded"
    return cr


def _f64(bits):
    return oracle.bf16_bits_to_f64(bits)


@pytest.mark.parametrize("T,out,r", [
    (300, 520, 40),      # ragged tokens and outputs against 128 x 256 tiles; K below one 64-block
    (128, 256, 8),       # one tile exactly
    (1000, 1032, 384),   # several tiles, ragged output tile of 8 columns, 6 K blocks per part
    (77, 8, 16),         # one partial tile
    (513, 4096, 768),    # many output tiles, a single-row last token tile
    (1, 264, 64),        # one token
])
def test_lora_form(T, out, r, layout):
    d = _layer(T, 16, out, r, 9500 + T + out + r)
    y = run_lora(d)
    assert_no_device_error()
    ref = oracle.compose_lora_fwd(_f64(d["base"]), _f64(d["xa"]), d["B"], d["g"], d["s"])
    _check("y (lora form)", y, ref)


@pytest.mark.parametrize("T,out,r", [
    (300, 520, 40),      # ragged tokens and outputs; K below one 64-block
    (128, 256, 8),       # one tile exactly
    (1000, 1032, 384),   # several tiles, ragged output tile; K = 3 x 128 on pairs
    (77, 8, 16),         # one partial tile
    (513, 4096, 776),    # many output tiles; K ragged against the 128-wide pair stages
    (1, 264, 64),        # one token
])
def test_lora_form_bf16_b(T, out, r, layout):
    d = _layer(T, 16, out, r, 9550 + T + out + r)
    y = run_lora_bf16(d)
    assert_no_device_error()
    _check("y (lora form, bf16 B)", y, ref_lora_bf16(d))


@pytest.mark.parametrize("T,inp,out,r", [
    (300, 264, 520, 40),     # ragged everything; K = 264 + 2 x 40
    (257, 1032, 776, 128),   # K blocks ragged in the x segment
    (128, 64, 256, 8),       # one tile, one K block per segment
    (1, 8, 8, 8),            # the smallest legal shape
    (640, 4096, 1024, 64),   # long K
    (200, 520, 4104, 24),    # 17 output tiles, the last one 8 columns wide
])
def test_linear_form(T, inp, out, r, layout):
    d = _layer(T, inp, out, r, 9600 + T + inp + out + r)
    y = run_linear(d)
    assert_no_device_error()
    ref = oracle.linear_fwd(_f64(d["x"]), _f64(d["W0"]), _f64(d["xa"]), d["B"], d["g"], d["s"])
    _check("y (linear form)", y, ref)


def _drawn(k):
    # a seeded draw over the accepted shapes (out, r and in multiples of 8)
    rng = np.random.default_rng(20261204 + k)
    return (int(rng.integers(1, 700)), 8 * int(rng.integers(1, 161)), 8 * int(rng.integers(1, 201)),
            8 * int(rng.integers(1, 97)))


@pytest.mark.parametrize("k", range(12))
def test_drawn_shapes_both_forms(k, layout):
    T, inp, out, r = _drawn(k)
    d = _layer(T, inp, out, r, 9800 + k)
    y = run_lora(d)
    assert_no_device_error()
    _check("y (lora form)", y, oracle.compose_lora_fwd(_f64(d["base"]), _f64(d["xa"]), d["B"], d["g"], d["s"]))
    y = run_linear(d)
    assert_no_device_error()
    _check("y (linear form)", y,
           oracle.linear_fwd(_f64(d["x"]), _f64(d["W0"]), _f64(d["xa"]), d["B"], d["g"], d["s"]))
    y = run_lora_bf16(d)
    assert_no_device_error()
    _check("y (lora form, bf16 B)", y, ref_lora_bf16(d))


def test_bitwise_reproducible(layout):
    d = _layer(300, 264, 520, 40, 9700)
    assert torch.equal(run_linear(d), run_linear(d))
    assert torch.equal(run_lora(d), run_lora(d))
    assert torch.equal(run_lora_bf16(d), run_lora_bf16(d))


def test_g_one_and_zero_adapter_lora_form_returns_base():
    # B = 0 and g = 1: y = base + 0 * base + 1 * 0 = base exactly
    d = _layer(300, 16, 520, 40, 9701)
    d["B"] = np.zeros_like(d["B"])
    d["g"] = np.ones_like(d["g"])
    y = run_lora(d)
    assert torch.equal(y, act_to_dev(d["base"]))
    assert torch.equal(run_lora_bf16(d), act_to_dev(d["base"]))


def test_full_size_sampled():
    # the high-rank layer: T = 15360 tokens, out = in = 8192, r = 384; sampled rows
    sh = wl.shape("high_rank")
    d = wl.make_layer(sh, wl.seed_for("high_rank") + 77)
    rows = np.sort(np.random.default_rng(9702).choice(sh.T, 48, replace=False))
    rows[-1] = sh.T - 1
    y_lin = to_f64(run_linear(d))[rows]
    ref_lin = oracle.linear_fwd(_f64(d["x"][rows]), _f64(d["W0"]), _f64(d["xa"][rows]), d["B"], d["g"], d["s"])
    y_lora = to_f64(run_lora(d))[rows]
    ref_lora = oracle.compose_lora_fwd(_f64(d["base"][rows]), _f64(d["xa"][rows]), d["B"], d["g"], d["s"])
    y_lb = to_f64(run_lora_bf16(d))[rows]
    ref_lb = ref_lora_bf16(d, rows)
    assert_no_device_error()
    for name, got, ref in (("y (linear form)", y_lin, ref_lin), ("y (lora form)", y_lora, ref_lora),
                           ("y (lora form, bf16 B)", y_lb, ref_lb)):
        check_bf16_rule(name, got, ref)
        cr = float(np.mean(got == oracle.bf16_bits_to_f64(oracle.f64_to_bf16_bits(ref))))
        assert cr >= CR_MIN, f"{name}: only {cr:.4f} of outputs correctly rounded"

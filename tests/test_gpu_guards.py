"""Out-of-bounds write checks without a sanitizer: every output and workspace
buffer is the middle of a larger allocation whose slack before and after is
filled with a sentinel; after each call the slack must be untouched.  Shapes
are ragged on purpose (partial M tiles, K tails, odd token counts, scalar and
vector compose paths)."""
import numpy as np
import pytest
import torch

import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import DEV, act_to_dev, assert_no_device_error, f32_dev

pytestmark = pytest.mark.gpu

SLACK = 4096            # bytes of guard before and after each buffer
SENTINEL = 0xA5


class Guarded:
    """A device buffer of `nbytes` with guarded slack; .view(dtype, shape)."""

    def __init__(self, nbytes, align=256):
        self.nbytes = nbytes
        self.raw = torch.full((SLACK + nbytes + SLACK + align,), SENTINEL, dtype=torch.uint8, device=DEV)
        base = self.raw.data_ptr()
        off = (-(base + SLACK)) % align
        self.lo = off + SLACK
        self.inner = self.raw[self.lo:self.lo + nbytes]

    def view(self, dtype, shape):
        return self.inner.view(dtype).view(*shape)

    def check(self, name):
        before = self.raw[self.lo - SLACK:self.lo]
        after = self.raw[self.lo + self.nbytes:self.lo + self.nbytes + SLACK]
        assert bool((before == SENTINEL).all()), f"{name}: write before the buffer"
        assert bool((after == SENTINEL).all()), f"{name}: write after the buffer"


@pytest.mark.parametrize("out,inp,r", [(257, 100, 17), (1000, 1040, 384), (130, 64, 768), (64, 2048, 48)])
def test_norm_writes_stay_in_bounds(out, inp, r):
    sh = wl.shape("high_rank", out=out, inp=inp, r=r, T=8)
    w = wl.make_weights(sh, 31)
    W0, A, B, m = (f32_dev(w[k]) for k in ("W0", "A", "B", "m"))
    norm_b, g_b = Guarded(out * 4), Guarded(out * 4)
    nbytes = dora.dora_norm_factored_workspace(out, inp, r)
    ws_b = Guarded(nbytes)
    norm, g = norm_b.view(torch.float32, (out,)), g_b.view(torch.float32, (out,))
    dora.dora_norm_factored(W0, A, B, m, w["s"], norm, g, ws_b.view(torch.uint8, (nbytes,)))
    torch.cuda.synchronize()
    norm_b.check("norm")
    g_b.check("g")
    ws_b.check("workspace")
    assert bool(torch.isfinite(norm).all())
    assert_no_device_error()


@pytest.mark.parametrize("act,T,out", [("bf16", 37, 104), ("bf16", 33, 101), ("f32", 29, 100), ("bf16", 300, 8192)])
def test_compose_writes_stay_in_bounds(act, T, out):
    rng = np.random.default_rng(T + out)
    f = {k: rng.standard_normal((T, out)).astype(np.float32) for k in ("base", "lora", "dy")}
    if act == "bf16":
        f = {k: wl.f32_to_bf16_bits(v) for k, v in f.items()}
    base, lora, dy = (act_to_dev(f[k]) for k in ("base", "lora", "dy"))
    esz = base.element_size()
    g = f32_dev(1 + 0.01 * rng.standard_normal(out))
    n = f32_dev(rng.uniform(0.5, 2.0, out))
    bufs = {k: Guarded(T * out * esz) for k in ("y", "db", "dl")}
    dm_b = Guarded(out * 4)
    wsn = dora.dora_compose_bwd_workspace(T, out)
    ws_b = Guarded(wsn)
    y, db, dl = (bufs[k].view(base.dtype, (T, out)) for k in ("y", "db", "dl"))
    dm = dm_b.view(torch.float32, (out,))
    dora.dora_compose_fwd(base, lora, g, 1.3, y)
    dora.dora_compose_bwd(dy, base, lora, g, n, 1.3, db, dl, dm, ws_b.view(torch.uint8, (wsn,)))
    torch.cuda.synchronize()
    for k, b in bufs.items():
        b.check(k)
    dm_b.check("d_mag")
    ws_b.check("workspace")
    assert_no_device_error()


@pytest.mark.parametrize("out,inp,r", [(257, 100, 17), (1000, 1040, 384), (130, 64, 768), (1030, 136, 64)])
def test_norm_gradient_writes_stay_in_bounds(out, inp, r):
    sh = wl.shape("high_rank", out=out, inp=inp, r=r, T=8)
    w = wl.make_weights(sh, 32)
    W0, A, B, m = (f32_dev(w[k]) for k in ("W0", "A", "B", "m"))
    norm = torch.empty(out, device=DEV)
    g = torch.empty(out, device=DEV)
    ws = torch.empty(dora.dora_norm_factored_workspace(out, inp, r), dtype=torch.uint8, device=DEV)
    dora.dora_norm_factored(W0, A, B, m, w["s"], norm, g, ws)
    dm = f32_dev(np.random.default_rng(out).standard_normal(out))
    dA_b, dB_b = Guarded(r * inp * 4), Guarded(out * r * 4)
    nbytes = dora.dora_norm_factored_bwd_workspace(out, inp, r)
    ws_b = Guarded(nbytes)
    dA, dB = dA_b.view(torch.float32, (r, inp)), dB_b.view(torch.float32, (out, r))
    dora.dora_norm_factored_bwd(W0, A, B, norm, g, dm, w["s"], dA, dB, ws_b.view(torch.uint8, (nbytes,)))
    torch.cuda.synchronize()
    dA_b.check("dA")
    dB_b.check("dB")
    ws_b.check("workspace")
    assert bool(torch.isfinite(dA).all()) and bool(torch.isfinite(dB).all())
    assert_no_device_error()


@pytest.mark.parametrize("T,inp,out,r", [(300, 264, 520, 40), (77, 8, 8, 16), (129, 1032, 776, 128)])
def test_fused_forward_writes_stay_in_bounds(T, inp, out, r):
    sh = wl.shape("high_rank", T=T, inp=inp, out=out, r=r)
    d = wl.make_layer(sh, 33)
    x, W0, xa, base = (act_to_dev(d[k]) for k in ("x", "W0", "xa", "base"))
    B, g = f32_dev(d["B"]), f32_dev(d["g"])
    B16 = act_to_dev(wl.f32_to_bf16_bits(d["B"]))
    nbytes = dora.dora_compose_fused_workspace(out, r)
    for form in ("lora", "lora_bf16", "linear"):
        y_b, ws_b = Guarded(T * out * 2), Guarded(nbytes)
        y = y_b.view(torch.bfloat16, (T, out))
        ws = ws_b.view(torch.uint8, (nbytes,))
        if form == "lora":
            dora.dora_compose_lora_fwd(base, xa, B, g, d["s"], y, ws)
        elif form == "lora_bf16":
            dora.dora_compose_lora_fwd_bf16(base, xa, B16, g, d["s"], y)
        else:
            dora.dora_linear_fwd(x, W0, xa, B, g, d["s"], y, ws)
        torch.cuda.synchronize()
        y_b.check(f"y ({form})")
        ws_b.check(f"workspace ({form})")
        assert bool(torch.isfinite(y.float()).all())
    assert_no_device_error()

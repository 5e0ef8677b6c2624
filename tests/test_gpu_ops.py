"""The torch.library ops and their autograd give bitwise the results of the
direct C-ABI calls (they only allocate and call the library)."""
import numpy as np
import pytest
import torch

import parameter_efficient_fine_gb300.ops as ops
from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import act_to_dev, assert_no_device_error, f32_dev, run_bwd, run_fwd, run_norm

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_ops_match_direct_calls_and_autograd(act):
    sh = wl.shape("high_rank", out=264, inp=384, r=40, T=96)
    d = wl.make_module(sh, 4242)
    s = d["s"]
    W0, A, B, m = (f32_dev(d[k]) for k in ("W0", "A", "B", "m"))
    if act == "bf16":
        base, lora, dy = (act_to_dev(d[k]) for k in ("base", "lora", "dy"))
    else:
        rng = np.random.default_rng(5)
        base, lora, dy = (f32_dev(rng.standard_normal((sh.T, sh.out)).astype(np.float32)) for _ in range(3))

    norm_d, g_d = run_norm(W0, A, B, m, s)
    norm_o, g_o = torch.ops.dora.norm_factored(W0, A, B, m, s)
    assert torch.equal(norm_o, norm_d) and torch.equal(g_o, g_d)

    y_d = run_fwd(base, lora, g_d, s)
    db_d, dl_d, dm_d = run_bwd(dy, base, lora, g_d, norm_d, s)

    base_a = base.clone().requires_grad_(True)
    lora_a = lora.clone().requires_grad_(True)
    m_a = m.clone().requires_grad_(True)
    y_o = ops.dora_module(base_a, lora_a, W0, A, B, m_a, s)
    assert torch.equal(y_o, y_d)
    y_o.backward(dy)
    assert torch.equal(base_a.grad, db_d)
    assert torch.equal(lora_a.grad, dl_d)
    assert torch.equal(m_a.grad, dm_d)
    assert_no_device_error()


def test_opcheck():
    sh = wl.shape("high_rank", out=128, inp=64, r=8, T=32)
    d = wl.make_module(sh, 77)
    s = d["s"]
    W0, A, B, m = (f32_dev(d[k]) for k in ("W0", "A", "B", "m"))
    base, lora, dy = (act_to_dev(d[k]) for k in ("base", "lora", "dy"))
    checks = ("test_schema", "test_autograd_registration", "test_faketensor")
    torch.library.opcheck(torch.ops.dora.norm_factored.default, (W0, A, B, m, s), test_utils=checks)
    norm, g = torch.ops.dora.norm_factored(W0, A, B, m, s)
    base_a = base.clone().requires_grad_(True)
    m_a = m.clone().requires_grad_(True)
    torch.library.opcheck(torch.ops.dora.compose.default, (base_a, lora, m_a, g, norm, s), test_utils=checks)
    torch.library.opcheck(torch.ops.dora.compose_bwd.default, (dy, base, lora, g, norm, s), test_utils=checks)
    assert_no_device_error()


def test_bf16_ops_match_direct_calls():
    from test_gpu_bf16 import _dev16, _module, run_norm_bf16
    sh = wl.shape("high_rank", out=264, inp=384, r=40, T=8)
    w, (w0b, ab, bb), _ = _module(sh, 4243)
    W0, A, B, m = _dev16(w0b), _dev16(ab), _dev16(bb), f32_dev(w["m"])
    n0_d, norm_d, g_d = run_norm_bf16(W0, A, B, m, w["s"])
    n0_o = torch.ops.dora.row_sumsq(W0)
    norm_o, g_o = torch.ops.dora.norm_factored_bf16(W0, A, B, m, n0_o, w["s"])
    assert torch.equal(n0_o, n0_d) and torch.equal(norm_o, norm_d) and torch.equal(g_o, g_d)
    assert_no_device_error()


def test_module_without_detach_matches_direct_calls():
    # the norm is NOT detached: gradients reach A and B through it, and every
    # gradient equals the direct C-ABI calls bitwise
    from test_gpu_norm_grad import run_norm_bwd
    sh = wl.shape("high_rank", out=264, inp=384, r=40, T=96)
    d = wl.make_module(sh, 4244)
    s = d["s"]
    W0, A, B, m = (f32_dev(d[k]) for k in ("W0", "A", "B", "m"))
    base, lora, dy = (act_to_dev(d[k]) for k in ("base", "lora", "dy"))
    norm_d, g_d = run_norm(W0, A, B, m, s)
    y_d = run_fwd(base, lora, g_d, s)
    db_d, dl_d, dm_d = run_bwd(dy, base, lora, g_d, norm_d, s)
    dA_d, dB_d = run_norm_bwd(W0, A, B, norm_d, g_d, dm_d, s)

    base_a, lora_a, A_a, B_a, m_a = (t.clone().requires_grad_(True) for t in (base, lora, A, B, m))
    y = ops.dora_module(base_a, lora_a, W0, A_a, B_a, m_a, s, detach_norm=False)
    assert torch.equal(y, y_d)
    y.backward(dy)
    assert torch.equal(base_a.grad, db_d) and torch.equal(lora_a.grad, dl_d) and torch.equal(m_a.grad, dm_d)
    assert torch.equal(A_a.grad, dA_d) and torch.equal(B_a.grad, dB_d)

    # with the norm detached (the default) no gradient reaches A or B
    A_b, B_b = A.clone().requires_grad_(True), B.clone().requires_grad_(True)
    base_b = base.clone().requires_grad_(True)
    ops.dora_module(base_b, lora, W0, A_b, B_b, m, s).backward(dy)
    assert A_b.grad is None and B_b.grad is None
    assert_no_device_error()


def test_opcheck_norm_grad_ops():
    sh = wl.shape("high_rank", out=128, inp=64, r=8, T=32)
    d = wl.make_module(sh, 78)
    s = d["s"]
    W0, A, B, m = (f32_dev(d[k]) for k in ("W0", "A", "B", "m"))
    base, lora, _ = (act_to_dev(d[k]) for k in ("base", "lora", "dy"))
    norm, g = torch.ops.dora.norm_factored(W0, A, B, m, s)
    dm = torch.randn_like(m)
    checks = ("test_schema", "test_autograd_registration", "test_faketensor")
    torch.library.opcheck(torch.ops.dora.norm_factored_bwd.default, (W0, A, B, norm, g, dm, s), test_utils=checks)
    A_a, B_a, m_a = (t.clone().requires_grad_(True) for t in (A, B, m))
    base_a = base.clone().requires_grad_(True)
    torch.library.opcheck(torch.ops.dora.module.default, (base_a, lora, W0, A_a, B_a, m_a, s), test_utils=checks)
    assert_no_device_error()

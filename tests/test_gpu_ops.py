"""The torch.library ops (the integration the method's page describes: the
kernels wrapped as a custom op that compiles without graph breaks).

Two kinds of check:
  * against the fp64 oracle: one DoRA module through ops.dora_module, forward
    and autograd backward, eagerly and under torch.compile(fullgraph=True)
    (a graph break raises), with the norm detached (the page's backward:
    d_base, d_lora, d_mag) and not detached (also dA, dB through the norm);
  * bitwise against the direct C-ABI calls (the ops only allocate and call
    the library), plus torch.library.opcheck of schemas, fake tensors and
    autograd registration.

Tolerances for the oracle checks, end to end: y, d_base, d_lora and d_mag
follow the bf16 rule of tests/gpu_util.py (bf16 activations) or the fp32
bounds of the parity tests widened by g's 1e-5 relative error (fp32
activations).  dA and dB come from the module's own n, g and d_mag, each
within 1e-5 relative of the oracle's (d_mag within its fp32 summation bound);
dA and dB are linear in c = g d_mag / n, so their normwise error is held to
4e-5 (three inputs at 1e-5 plus the gradient's own 1e-5).
"""
import numpy as np
import pytest
import torch

import oracle
import parameter_efficient_fine_gb300.ops as ops
from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import (act_to_dev, act_to_f64, assert_no_device_error, check_bf16_rule, check_bound, check_rel,
                      dmag_bound, f32_dev, run_bwd, run_fwd, run_norm, to_f64)

GRAD_FRO_REL = 4e-5

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


# ---------------------------------------------------------------------------
# against the oracle, eager and compiled
# ---------------------------------------------------------------------------
def _module_case(act, seed):
    sh = wl.shape("high_rank", out=264, inp=384, r=40, T=96)
    d = wl.make_module(sh, seed)
    if act == "f32":
        rng = np.random.default_rng(seed + 1)
        for k in ("base", "lora", "dy"):
            d[k] = rng.standard_normal((sh.T, sh.out)).astype(np.float32)
        d["lora"] *= np.float32(np.sqrt(sh.r) * sh.sigma_B)
    return sh, d


def _oracle_refs(d):
    s = d["s"]
    n_ref, g_ref = oracle.weight_norm(d["W0"], d["A"], d["B"], d["m"], s)
    b64, l64, d64 = (act_to_f64(d[k]) for k in ("base", "lora", "dy"))
    y_ref = oracle.compose_fwd(b64, l64, g_ref, s)
    db_ref, dl_ref, dm_ref = oracle.compose_bwd(d64, b64, l64, g_ref, n_ref, s)
    dA_ref, dB_ref = oracle.norm_grad(d["W0"], d["A"], d["B"], s, n_ref, g_ref, dm_ref)
    return dict(n=n_ref, g=g_ref, y=y_ref, db=db_ref, dl=dl_ref, dm=dm_ref, dA=dA_ref, dB=dB_ref,
                b64=b64, l64=l64, d64=d64)


def _check_act(name, got, ref, act, ref_abs):
    if act == "bf16":
        check_bf16_rule(name, got, ref)
    else:
        check_bound(name, got, ref, 2.0 ** -21 * ref_abs + 1.1e-5 * np.abs(ref))


def _check_module(act, d, ref, y, base_a, lora_a, m_a, A_a=None, B_a=None):
    s = d["s"]
    b64, l64, d64, g = ref["b64"], ref["l64"], ref["d64"], ref["g"]
    _check_act("y", to_f64(y), ref["y"], act, np.abs(b64) + np.abs(g) * s * np.abs(l64))
    gd = np.abs(g)[None, :] * np.abs(d64)
    _check_act("d_base", to_f64(base_a.grad), ref["db"], act, gd)
    _check_act("d_lora", to_f64(lora_a.grad), ref["dl"], act, gd * (1 + s))
    dm = to_f64(m_a.grad)
    check_bf16_rule("d_mag", dm, ref["dm"])
    check_bound("d_mag", dm, ref["dm"], dmag_bound(d64, b64, l64, ref["n"], s) + 1.1e-5 * np.abs(ref["dm"]))
    if A_a is not None:
        for name, got, want in (("dA", A_a.grad, ref["dA"]), ("dB", B_a.grad, ref["dB"])):
            got = to_f64(got)
            assert np.all(np.isfinite(got)), name
            fro = float(np.linalg.norm(got - want) / np.linalg.norm(want))
            assert fro <= GRAD_FRO_REL, f"{name}: ||err||/||ref|| = {fro:.3e}"
    else:
        assert A_a is None and B_a is None


def _leaves(d, act, detach_norm):
    W0 = f32_dev(d["W0"])
    A, B, m = (f32_dev(d[k]) for k in ("A", "B", "m"))
    base, lora, dy = (act_to_dev(d[k]) for k in ("base", "lora", "dy"))
    base_a, lora_a, m_a = (t.clone().requires_grad_(True) for t in (base, lora, m))
    if not detach_norm:
        A, B = A.clone().requires_grad_(True), B.clone().requires_grad_(True)
    return W0, A, B, base_a, lora_a, m_a, dy


@pytest.mark.parametrize("detach_norm", [True, False])
@pytest.mark.parametrize("act", ["bf16", "f32"])
def test_module_eager_against_oracle(act, detach_norm):
    sh, d = _module_case(act, 4301 + (0 if detach_norm else 1))
    ref = _oracle_refs(d)
    W0, A, B, base_a, lora_a, m_a, dy = _leaves(d, act, detach_norm)
    y = ops.dora_module(base_a, lora_a, W0, A, B, m_a, d["s"], detach_norm=detach_norm)
    y.backward(dy)
    torch.cuda.synchronize()
    _check_module(act, d, ref, y, base_a, lora_a, m_a, *(() if detach_norm else (A, B)))
    # the norm op alone
    norm, g = torch.ops.dora.norm_factored(W0, A.detach(), B.detach(), m_a.detach(), d["s"])
    check_rel("norm", to_f64(norm), ref["n"])
    check_rel("g", to_f64(g), ref["g"])
    assert_no_device_error()


@pytest.mark.parametrize("backend", ["aot_eager", "inductor"])
@pytest.mark.parametrize("detach_norm", [True, False])
def test_module_compiled_fullgraph_against_oracle(backend, detach_norm):
    # fullgraph=True makes any graph break an error; the compiled forward and
    # backward then go through the same ops and must meet the oracle bar
    torch._dynamo.reset()
    act = "bf16"
    sh, d = _module_case(act, 4311 + (0 if detach_norm else 1))
    ref = _oracle_refs(d)
    s = d["s"]
    W0, A, B, base_a, lora_a, m_a, dy = _leaves(d, act, detach_norm)

    def layer(base, lora, W0, A, B, m):
        return ops.dora_module(base, lora, W0, A, B, m, s, detach_norm=detach_norm)

    explain = torch._dynamo.explain(layer)(base_a, lora_a, W0, A, B, m_a)
    assert explain.graph_break_count == 0 and explain.graph_count == 1, explain.break_reasons
    torch._dynamo.reset()
    compiled = torch.compile(layer, fullgraph=True, backend=backend)
    y = compiled(base_a, lora_a, W0, A, B, m_a)
    y.backward(dy)
    torch.cuda.synchronize()
    _check_module(act, d, ref, y, base_a, lora_a, m_a, *(() if detach_norm else (A, B)))
    # and bitwise what the eager ops give on the same inputs
    W0e, Ae, Be, base_e, lora_e, m_e, _ = _leaves(d, act, detach_norm)
    ye = ops.dora_module(base_e, lora_e, W0e, Ae, Be, m_e, s, detach_norm=detach_norm)
    ye.backward(dy)
    assert torch.equal(y, ye)
    assert torch.equal(base_a.grad, base_e.grad) and torch.equal(m_a.grad, m_e.grad)
    if not detach_norm:
        assert torch.equal(A.grad, Ae.grad) and torch.equal(B.grad, Be.grad)
    assert_no_device_error()

"""Failure detection without a GPU fault: the kernels' waits on on-chip
barriers are bounded.  A test hook makes the norm kernels withhold their loads,
so those waits expire after a short limit; the kernels must record the failure
in the device error word, release their resources and exit, and the context
must stay usable for a correct call right after."""
import numpy as np
import pytest

import oracle
import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import assert_no_device_error, check_rel, f32_dev, run_norm, to_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("out,inp,r", [(256, 64, 16), (256, 64, 384)])
def test_expired_wait_is_reported_and_context_survives(out, inp, r):
    sh = wl.shape("high_rank", out=out, inp=inp, r=r, T=8)
    w = wl.make_weights(sh, 5)
    W0, A, B, m = (f32_dev(w[k]) for k in ("W0", "A", "B", "m"))
    assert_no_device_error()
    dora.dora_test_stall_loads(True, 50_000_000)      # 50 ms
    try:
        run_norm(W0, A, B, m, w["s"])
        code = dora.dora_device_error()                # synchronises
    finally:
        dora.dora_test_stall_loads(False)
    assert code != 0
    # the same call now completes and is correct
    norm, g = run_norm(W0, A, B, m, w["s"])
    n_ref, g_ref = oracle.weight_norm(w["W0"], w["A"], w["B"], w["m"], w["s"])
    check_rel("norm", to_f64(norm), n_ref)
    check_rel("g", to_f64(g), g_ref)
    assert_no_device_error()


def _stalled(call):
    assert_no_device_error()
    dora.dora_test_stall_loads(True, 50_000_000)      # 50 ms
    try:
        call()
        code = dora.dora_device_error()                # synchronises
    finally:
        dora.dora_test_stall_loads(False)
    return code


def test_norm_gradient_expired_wait_is_reported():
    from test_gpu_norm_grad import run_norm_bwd
    sh = wl.shape("high_rank", out=300, inp=256, r=40, T=8)
    w = wl.make_weights(sh, 6)
    W0, A, B, m = (f32_dev(w[k]) for k in ("W0", "A", "B", "m"))
    norm, g = run_norm(W0, A, B, m, w["s"])
    dm = f32_dev(np.random.default_rng(6).standard_normal(sh.out).astype(np.float32))
    assert _stalled(lambda: run_norm_bwd(W0, A, B, norm, g, dm, w["s"])) != 0
    dA, dB = run_norm_bwd(W0, A, B, norm, g, dm, w["s"])
    dA_ref, dB_ref = oracle.norm_grad(w["W0"], w["A"], w["B"], w["s"], to_f64(norm), to_f64(g), to_f64(dm))
    assert np.linalg.norm(to_f64(dA) - dA_ref) <= 1e-5 * np.linalg.norm(dA_ref)
    assert np.linalg.norm(to_f64(dB) - dB_ref) <= 1e-5 * np.linalg.norm(dB_ref)
    assert_no_device_error()


@pytest.mark.parametrize("form", ["lora", "linear"])
def test_fused_forward_expired_wait_is_reported(form):
    # the lora form's epilogue warps have base copies in flight when the
    # MMA-side waits expire: they must drain them before leaving
    from gpu_util import check_bf16_rule
    from test_gpu_fused import _f64, _layer, run_linear, run_lora
    d = _layer(300, 264, 520, 40, 9800)
    run = run_lora if form == "lora" else run_linear
    assert _stalled(lambda: run(d)) != 0
    y = to_f64(run(d))
    if form == "lora":
        ref = oracle.compose_lora_fwd(_f64(d["base"]), _f64(d["xa"]), d["B"], d["g"], d["s"])
    else:
        ref = oracle.linear_fwd(_f64(d["x"]), _f64(d["W0"]), _f64(d["xa"]), d["B"], d["g"], d["s"])
    check_bf16_rule("y", y, ref)
    assert_no_device_error()

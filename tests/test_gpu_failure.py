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

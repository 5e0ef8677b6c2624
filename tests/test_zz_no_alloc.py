"""The allocation-free compose backward, dora_compose_bwd_noalloc.

Some callers cannot allocate device memory where they run the backward -- code
embedded in an application that owns a fixed device memory pool and exposes no
allocator, or services that forbid cudaMalloc after start-up because it
synchronises the device.  For them the library keeps the d_mag partial sums in
one fixed device array instead of a caller workspace.  This test calls that
entry point through the C ABI twice in a row (the second call finds the first
call's leftovers in the shared array) and checks each result against the fp64
oracle under the usual GPU tolerances, and against the workspace entry point
dora_compose_bwd, which launches the same grid and so must agree bitwise.  It
is collected last so that a failure here cannot hide the other tests' results.
"""
import numpy as np
import pytest
import torch

import oracle
import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import (DEV, act_to_dev, act_to_f64, assert_no_device_error, check_bf16_rule, check_bound,
                      dmag_bound, f32_dev, run_bwd, to_f64)

pytestmark = pytest.mark.gpu


def _inputs(out, T, seed):
    sh = wl.shape("high_rank", out=out, inp=64, r=16, T=T)
    a = wl.make_activations(sh, seed)
    rng = np.random.default_rng(seed)
    g = (1 + rng.uniform(-0.05, 0.05, out)).astype(np.float32)
    n = rng.uniform(0.5, 2.0, out).astype(np.float32)
    return a, g, n, sh.s


def test_noalloc_backward_matches_oracle_and_workspace_entry_point_twice():
    for out, T, seed in ((4096, 1536, 1), (1000, 333, 2)):
        a, g, n, s = _inputs(out, T, seed)
        dy, base, lora = (act_to_dev(a[k]) for k in ("dy", "base", "lora"))
        gd, nd = f32_dev(g), f32_dev(n)
        db_ref, dl_ref, dm_ref = run_bwd(dy, base, lora, gd, nd, s)
        db = torch.empty_like(dy)
        dl = torch.empty_like(dy)
        dm = torch.full((out,), float("nan"), device=DEV)
        dora.dora_compose_bwd_noalloc(dy, base, lora, gd, nd, s, db, dl, dm)
        torch.cuda.synchronize()
        # the fp64 oracle on the same inputs
        d64, b64, l64 = (act_to_f64(a[k]) for k in ("dy", "base", "lora"))
        g64, n64 = g.astype(np.float64), n.astype(np.float64)
        db_o, dl_o, dm_o = oracle.compose_bwd(d64, b64, l64, g64, n64, s)
        check_bf16_rule("d_base", to_f64(db), db_o)
        check_bf16_rule("d_lora", to_f64(dl), dl_o)
        check_bf16_rule("d_mag", to_f64(dm), dm_o)
        check_bound("d_mag", to_f64(dm), dm_o, dmag_bound(d64, b64, l64, n64, s))
        # the workspace entry point: same grid, same summation order
        assert torch.equal(db, db_ref) and torch.equal(dl, dl_ref)
        assert torch.equal(dm.view(torch.int32), dm_ref.view(torch.int32))
    assert_no_device_error()


def test_noalloc_rejects_rows_wider_than_the_scratch():
    lib = dora.load_library()
    too_wide = (1 << 20) + 8     # DORA_NOALLOC_SCRATCH_FLOATS + 8 columns
    p = 1 << 20                  # never dereferenced: the call returns before any launch
    st = lib.dora_compose_bwd_noalloc(1, p, p, p, p, p, 1.0, 4, too_wide, p, p, p, None)
    assert st == 2               # DORA_ERR_SHAPE

"""bf16 weights: dora_row_sumsq_bf16 and dora_norm_factored_bf16 against the
fp64 oracle, which forms W0 + s B A densely from the same bf16 values (upcast
exactly).  Tolerance: norm and g relative error <= 1e-5 (the fp32 rule)."""
import numpy as np
import pytest
import torch

import oracle
import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import DEV, assert_no_device_error, check_rel, f32_dev, to_f64

pytestmark = pytest.mark.gpu


def _bf16(a):
    bits = wl.f32_to_bf16_bits(np.ascontiguousarray(a, dtype=np.float32))
    return bits, oracle.bf16_bits_to_f64(bits)


def _dev16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(DEV).view(torch.bfloat16)


def run_norm_bf16(W0, A, B, m, s):
    out, inp = W0.shape
    r = A.shape[0]
    n0sq = torch.empty(out, device=DEV)
    dora.dora_row_sumsq_bf16(W0, n0sq)
    norm = torch.empty(out, device=DEV)
    g = torch.empty(out, device=DEV)
    ws = torch.empty(max(dora.dora_norm_factored_bf16_workspace(out, inp, r), 1), dtype=torch.uint8, device=DEV)
    dora.dora_norm_factored_bf16(W0, A, B, m, n0sq, s, norm, g, ws)
    return n0sq, norm, g


def _module(sh, seed):
    w = wl.make_weights(sh, seed)
    (w0b, w0), (ab, a), (bb, b) = _bf16(w["W0"]), _bf16(w["A"]), _bf16(w["B"])
    return w, (w0b, ab, bb), (w0, a, b)


@pytest.mark.parametrize("out,inp,r", [
    (1000, 1040, 384),   # ragged M tile and K block, N = 256 + 128
    (300, 256, 1),       # r = 1: B padded to a 16-byte row
    (257, 512, 17),      # r not a multiple of 8
    (384, 256, 272),     # one N chunk of 272
    (200, 128, 400),     # two N chunks
    (130, 64, 768),      # two N chunks of 384
    (8, 8, 5),           # one K block, mostly out of bounds
    (1, 16, 2),          # a single row
    (300, 1040, 128),    # 64-wide K blocks with a tail
    (260, 200, 129),     # N = 144
])
def test_bf16_norm_matches_oracle(out, inp, r):
    sh = wl.shape("high_rank", out=out, inp=inp, r=r, T=8)
    w, (w0b, ab, bb), (w0, a, b) = _module(sh, 9100 + out + r)
    s = w["s"]
    n0sq, norm, g = run_norm_bf16(_dev16(w0b), _dev16(ab), _dev16(bb), f32_dev(w["m"]), s)
    n_ref, g_ref = oracle.weight_norm(w0, a, b, w["m"], s)
    check_rel("n0sq", to_f64(n0sq), np.sum(w0 * w0, axis=1), tol=2e-5)
    check_rel("norm", to_f64(norm), n_ref)
    check_rel("g", to_f64(g), g_ref)
    assert_no_device_error()


@pytest.mark.parametrize("k", range(10))
def test_bf16_norm_drawn_shapes(k):
    # a seeded draw over the accepted shapes (in a multiple of 8, any r and out)
    rng = np.random.default_rng(20261206 + k)
    out, inp, r = int(rng.integers(1, 1600)), 8 * int(rng.integers(1, 201)), int(rng.integers(1, 801))
    test_bf16_norm_matches_oracle(out, inp, r)


def test_bf16_zero_adapter_gives_unit_g():
    sh = wl.shape("high_rank", out=512, inp=1024, r=32, T=8)
    w, (w0b, ab, bb), (w0, a, b) = _module(sh, 5)
    bb = np.zeros_like(bb)
    m = np.sqrt(np.sum(w0 * w0, axis=1)).astype(np.float32)
    _, norm, g = run_norm_bf16(_dev16(w0b), _dev16(ab), _dev16(bb), f32_dev(m), w["s"])
    gh = to_f64(g)
    assert np.max(np.abs(gh - 1.0)) <= 4 * 2.0 ** -23
    assert_no_device_error()


@pytest.mark.parametrize("r", [16, 128, 384, 768])
def test_bf16_full_size_sampled_rows(r):
    sh = wl.shape("rank_sweep", r=r)
    w, (w0b, ab, bb), (w0, a, b) = _module(sh, 8800 + r)
    s = w["s"]
    W0, A, B, m = _dev16(w0b), _dev16(ab), _dev16(bb), f32_dev(w["m"])
    n0sq, norm, g = run_norm_bf16(W0, A, B, m, s)
    rng = np.random.default_rng(r)
    rows = np.unique(np.concatenate([rng.choice(sh.out, 256, replace=False), [0, sh.out - 1]]))
    n_ref, g_ref = oracle.weight_norm(w0[rows], a, b[rows], w["m"][rows], s)
    check_rel("norm", to_f64(norm)[rows], n_ref)
    check_rel("g", to_f64(g)[rows], g_ref)
    _, norm2, _ = run_norm_bf16(W0, A, B, m, s)
    assert torch.equal(norm.view(torch.int32), norm2.view(torch.int32))   # bitwise reproducible
    assert_no_device_error()


@pytest.mark.parametrize("out,inp,r", [(257, 128, 17), (1000, 1040, 384)])
def test_bf16_norm_writes_stay_in_bounds(out, inp, r):
    from test_gpu_guards import Guarded
    sh = wl.shape("high_rank", out=out, inp=inp, r=r, T=8)
    w, (w0b, ab, bb), _ = _module(sh, 31)
    W0, A, B, m = _dev16(w0b), _dev16(ab), _dev16(bb), f32_dev(w["m"])
    n0_b, norm_b, g_b = Guarded(out * 4), Guarded(out * 4), Guarded(out * 4)
    nbytes = dora.dora_norm_factored_bf16_workspace(out, inp, r)
    ws_b = Guarded(nbytes)
    n0 = n0_b.view(torch.float32, (out,))
    dora.dora_row_sumsq_bf16(W0, n0)
    dora.dora_norm_factored_bf16(W0, A, B, m, n0, w["s"], norm_b.view(torch.float32, (out,)),
                                 g_b.view(torch.float32, (out,)), ws_b.view(torch.uint8, (nbytes,)))
    torch.cuda.synchronize()
    for name, b in (("n0sq", n0_b), ("norm", norm_b), ("g", g_b), ("workspace", ws_b)):
        b.check(name)
    assert_no_device_error()

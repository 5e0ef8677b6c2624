"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
library through its C ABI, and compare with the fp64 oracle under the stated
tolerances.

Tolerances (stated once, used by every GPU test):
  * norm and g: relative error <= 1e-5 (fp32 result).
  * bf16 outputs and gradients (y, d_base, d_lora) and d_mag:
        |err| <= 2^-7 * |ref| + 1e-3 elementwise, cosine similarity >= 0.99999.
  * fp32 activations (the tiny workload): derived from the fp32 arithmetic of
    the kernel -- at most four roundings of magnitude <= |base| + |g s lora|
    when both sides use the same fp32 g:
        |err| <= 2^-21 * (|base| + |g| s |lora|)    (compose fwd)
        |err| <= 2^-22 * |g| (1 + s) |dy|           (d_base, d_lora)
    When g comes from the GPU norm instead, its 1e-5 relative error is added.
  * d_mag (any dtype), a rigorous fp32 summation bound: with at most T + 16
    sequential additions, |err| <= 2^-24 (T + 16) * sum_t |dy| (|base| + s|lora|) / n.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import workloads as wl

DEV = torch.device("cuda:0")
BF16_REL = 2.0 ** -7
BF16_ABS = 1e-3
NORM_REL = 1e-5
COS_MIN = 0.99999


def act_to_dev(a: np.ndarray, dev=DEV) -> torch.Tensor:
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def act_to_f64(a: np.ndarray) -> np.ndarray:
    if a.dtype == np.uint16:
        return oracle.bf16_bits_to_f64(a)
    return a.astype(np.float64)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def f32_dev(a: np.ndarray, dev=DEV) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def run_norm(W0, A, B, m, s, dev=DEV):
    """Inputs as device tensors; returns (norm, g) device tensors."""
    out, inp = W0.shape
    r = A.shape[0]
    norm = torch.empty(out, device=dev)
    g = torch.empty(out, device=dev)
    ws = torch.empty(max(dora.dora_norm_factored_workspace(out, inp, r), 1), dtype=torch.uint8, device=dev)
    dora.dora_norm_factored(W0, A, B, m, s, norm, g, ws)
    return norm, g


def run_fwd(base, lora, g, s):
    y = torch.empty_like(base)
    dora.dora_compose_fwd(base, lora, g, s, y)
    return y


def run_bwd(dy, base, lora, g, norm, s):
    T, out = dy.shape
    db = torch.empty_like(dy)
    dl = torch.empty_like(dy)
    dm = torch.empty(out, device=dy.device)
    ws = torch.empty(max(dora.dora_compose_bwd_workspace(T, out), 1), dtype=torch.uint8, device=dy.device)
    dora.dora_compose_bwd(dy, base, lora, g, norm, s, db, dl, dm, ws)
    return db, dl, dm


def assert_no_device_error():
    torch.cuda.synchronize()
    code = dora.dora_device_error()
    assert code == 0, f"a kernel wait gave up (code {code})"


def cosine(a, b) -> float:
    a = np.asarray(a, np.float64).ravel()
    b = np.asarray(b, np.float64).ravel()
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    if na == 0 and nb == 0:
        return 1.0
    return float(a @ b / (na * nb))


def check_rel(name, got, ref, tol=NORM_REL):
    rel = np.abs(got - ref) / np.abs(ref)
    worst = float(np.max(rel)) if rel.size else 0.0
    assert worst <= tol, f"{name}: max rel err {worst:.3e} > {tol:.1e}"
    return worst


def check_bf16_rule(name, got, ref, cos=True):
    err = np.abs(got - ref)
    bound = BF16_REL * np.abs(ref) + BF16_ABS
    bad = int(np.count_nonzero(err > bound))
    assert bad == 0, f"{name}: {bad} elements outside 2^-7|ref|+1e-3 (max err {float(err.max()):.3e})"
    if cos and ref.size > 1:
        c = cosine(got, ref)
        assert c >= COS_MIN, f"{name}: cosine {c:.8f} < {COS_MIN}"


def check_bound(name, got, ref, bound):
    err = np.abs(got - ref)
    bad = int(np.count_nonzero(err > bound))
    assert bad == 0, f"{name}: {bad} elements over the bound (worst ratio {float(np.max(err / np.maximum(bound, 1e-300))):.3f})"


def dmag_bound(dy, base, lora, n, s):
    T = dy.shape[0]
    mag = np.sum(np.abs(dy) * (np.abs(base) + s * np.abs(lora)), axis=0) / np.abs(n)
    return 2.0 ** -24 * (T + 16) * mag + 1e-30


def weights_dev(d):
    return tuple(f32_dev(d[k]) for k in ("W0", "A", "B", "m"))


def full_check(sh, seed, bwd=True):
    """Norm, forward and (optionally) backward of one module, all elements."""
    d = wl.make_module(sh, seed)
    s = d["s"]
    W0, A, B, m = weights_dev(d)
    norm, g = run_norm(W0, A, B, m, s)
    n_ref, g_ref = oracle.weight_norm(d["W0"], d["A"], d["B"], d["m"], s)
    check_rel("norm", to_f64(norm), n_ref)
    check_rel("g", to_f64(g), g_ref)

    base, lora, dy = (act_to_dev(d[k]) for k in ("base", "lora", "dy"))
    b64, l64, d64 = (act_to_f64(d[k]) for k in ("base", "lora", "dy"))
    y = run_fwd(base, lora, g, s)
    y_ref = oracle.compose_fwd(b64, l64, g_ref, s)
    if sh.act == "bf16":
        check_bf16_rule("y", to_f64(y), y_ref)
    else:
        bound = 2.0 ** -21 * (np.abs(b64) + np.abs(g_ref) * s * np.abs(l64)) + 1.1e-5 * np.abs(y_ref)
        check_bound("y", to_f64(y), y_ref, bound)
    if bwd:
        db, dl, dm = run_bwd(dy, base, lora, g, norm, s)
        db_ref, dl_ref, dm_ref = oracle.compose_bwd(d64, b64, l64, g_ref, n_ref, s)
        if sh.act == "bf16":
            check_bf16_rule("d_base", to_f64(db), db_ref)
            check_bf16_rule("d_lora", to_f64(dl), dl_ref)
        else:
            gb = np.abs(g_ref)[None, :] * np.abs(d64)
            check_bound("d_base", to_f64(db), db_ref, 2.0 ** -22 * gb + 1.1e-5 * np.abs(db_ref))
            check_bound("d_lora", to_f64(dl), dl_ref, 2.0 ** -22 * gb * (1 + s) + 1.1e-5 * np.abs(dl_ref))
        check_bf16_rule("d_mag", to_f64(dm), dm_ref)
        check_bound("d_mag", to_f64(dm), dm_ref, dmag_bound(d64, b64, l64, n_ref, s) + 1.1e-5 * np.abs(dm_ref))
    assert_no_device_error()

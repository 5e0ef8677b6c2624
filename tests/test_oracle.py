"""Pins for the fp64 oracle: checks against closed forms, library routines,
hand-computed fixtures, finite differences and invariants -- never against a
retyped copy of the oracle's own formulas.  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return np.max(np.abs(a - b) / np.maximum(np.abs(b), 1e-300))


# --------------------------------------------------------------------------
# bf16 encode / decode
# --------------------------------------------------------------------------

def test_bf16_decode_known_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0001, 0x7F7F, 0x8000, 0x3F81], np.uint16)
    want = [1.0, -2.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, -0.0, 1 + 2 ** -7]
    got = oracle.bf16_bits_to_f64(bits)
    assert np.array_equal(got, np.array(want))
    assert np.signbit(got[4])


def test_bf16_encode_matches_torch_on_binary32_inputs():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    parts = [
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-38).astype(np.float32),   # bf16 subnormals
        (rng.standard_normal(2000) * 1e30).astype(np.float32),
        rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ]
    x = np.concatenate(parts)
    x = x[np.isfinite(x)]
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, want)


def test_bf16_encode_single_rounding_from_fp64():
    # 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7: ties go to the even 1.0;
    # anything above the midpoint (even below binary32 resolution) rounds up.
    x = np.array([1 + 2 ** -8, 1 + 2 ** -8 + 2 ** -30, 1 + 3 * 2 ** -8,
                  1 + 3 * 2 ** -8 - 2 ** -40, -(1 + 2 ** -8 + 2 ** -30)])
    want = np.array([0x3F80, 0x3F81, 0x3F82, 0x3F81, 0xBF81], np.uint16)
    assert np.array_equal(oracle.f64_to_bf16_bits(x), want)


# --------------------------------------------------------------------------
# (a) weight norm
# --------------------------------------------------------------------------

def test_norm_hand_fixtures():
    for case in _load("norm_hand.json")["cases"]:
        n, g = oracle.weight_norm(np.array(case["W0"], float), np.array(case["A"], float),
                                  np.array(case["B"], float), np.array(case["m"], float), case["s"])
        assert _rel(n, case["n"]) < 1e-15
        assert _rel(g, case["g"]) < 1e-15


def test_norm_b_zero_is_library_row_norm_and_g_one():
    rng = np.random.default_rng(1)
    W0 = rng.standard_normal((37, 53))
    A = rng.standard_normal((5, 53))
    B = np.zeros((37, 5))
    ref = np.linalg.norm(W0, axis=1)
    n, g = oracle.weight_norm(W0, A, B, ref, 1.7)
    assert _rel(n, ref) < 1e-14
    assert np.max(np.abs(g - 1.0)) <= 4 * np.finfo(np.float64).eps


def _orthonormal_rows(rng, r, n):
    q, _ = np.linalg.qr(rng.standard_normal((n, r)))
    return q.T.copy()          # [r, n], rows orthonormal


def test_norm_pythagoras_closed_form():
    # W0 rows orthogonal to the row space of A, A rows orthonormal:
    # ||W0_i + s B_i A||^2 = ||W0_i||^2 + s^2 ||B_i||^2
    rng = np.random.default_rng(2)
    out, inp, r, s = 19, 40, 6, 2.5
    A = _orthonormal_rows(rng, r, inp)
    R = rng.standard_normal((out, inp))
    W0 = R - (R @ A.T) @ A
    B = rng.standard_normal((out, r))
    want = np.sqrt(np.sum(W0 ** 2, axis=1) + s * s * np.sum(B ** 2, axis=1))
    n = oracle.adapted_row_norm(W0, A, B, s)
    assert _rel(n, want) < 1e-13


def test_norm_parallel_rows_fix_cross_term_sign():
    # W0_i = lam_i * B_i A with orthonormal A: n_i = |lam_i + s| * ||B_i||.
    # A wrong sign on the cross term would give |lam_i - s| instead.
    rng = np.random.default_rng(3)
    out, inp, r, s = 11, 24, 4, 1.5
    A = _orthonormal_rows(rng, r, inp)
    B = rng.standard_normal((out, r))
    lam = np.linspace(-3 * s, 2 * s, out)
    W0 = lam[:, None] * (B @ A)
    want = np.abs(lam + s) * np.linalg.norm(B, axis=1)
    n = oracle.adapted_row_norm(W0, A, B, s)
    assert np.max(np.abs(n - want) / np.maximum(want, 1.0)) < 1e-13


def test_norm_is_per_output_row():
    # a joint permutation of the input columns of W0 and A leaves every row
    # norm unchanged; permuting output rows of (W0, B, m) permutes (n, g)
    rng = np.random.default_rng(4)
    out, inp, r, s = 16, 16, 3, 0.8
    W0 = rng.standard_normal((out, inp))
    A = rng.standard_normal((r, inp))
    B = rng.standard_normal((out, r))
    m = rng.uniform(0.5, 2.0, out)
    n, g = oracle.weight_norm(W0, A, B, m, s)
    pc = rng.permutation(inp)
    n2, _ = oracle.weight_norm(W0[:, pc], A[:, pc], B, m, s)
    assert _rel(n2, n) < 1e-14
    pr = rng.permutation(out)
    n3, g3 = oracle.weight_norm(W0[pr], A, B[pr], m[pr], s)
    assert _rel(n3, n[pr]) < 1e-14 and _rel(g3, g[pr]) < 1e-14


@pytest.mark.parametrize("out", [1, 2, 3, 7, 16])
@pytest.mark.parametrize("inp", [1, 2, 3, 7, 16])
@pytest.mark.parametrize("r", [1, 2, 5])
def test_norm_factored_identity_bruteforce(out, inp, r):
    # the page's base + cross + Gram split, evaluated in fp64 from U = W0 A^T
    # and G = A A^T, must reproduce the dense row norm
    rng = np.random.default_rng(100 * out + 10 * inp + r)
    W0 = rng.standard_normal((out, inp))
    A = rng.standard_normal((r, inp))
    B = rng.standard_normal((out, r))
    s = 0.7
    U = W0 @ A.T
    G = A @ A.T
    n2 = np.sum(W0 * W0, 1) + 2 * s * np.sum(U * B, 1) + s * s * np.einsum("ik,kl,il->i", B, G, B)
    n = oracle.adapted_row_norm(W0, A, B, s)
    assert np.max(np.abs(n * n - n2) / np.maximum(n * n, 1e-3)) < 1e-12


def test_norm_zero_row_gives_ieee_g():
    W0 = np.zeros((2, 4))
    A = np.ones((1, 4))
    B = np.zeros((2, 1))
    n, g = oracle.weight_norm(W0, A, B, np.array([1.0, 0.0]), 1.0)
    assert np.all(n == 0)
    assert np.isinf(g[0]) and np.isnan(g[1])


# --------------------------------------------------------------------------
# (b) compose forward / backward
# --------------------------------------------------------------------------

def test_compose_hand_fixture():
    c = _load("compose_hand.json")
    base, lora, g, n, s, dy = (np.array(c[k], float) for k in ("base", "lora", "g", "n", "s", "dy"))
    assert np.array_equal(oracle.compose_fwd(base, lora, g, s), np.array(c["y"]))
    assert np.array_equal(oracle.compose_fwd_stable(base, lora, g, s), np.array(c["y"]))
    db, dl, dm = oracle.compose_bwd(dy, base, lora, g, n, s)
    assert np.array_equal(db, np.array(c["d_base"]))
    assert np.array_equal(dl, np.array(c["d_lora"]))
    assert np.array_equal(dm, np.array(c["d_mag"]))


def test_compose_stable_equals_plain_in_fp64():
    rng = np.random.default_rng(6)
    T, out, s = 64, 48, 1.3
    base = rng.standard_normal((T, out))
    lora = rng.standard_normal((T, out)) * 0.2
    g = 1 + rng.uniform(-2 ** -9, 2 ** -9, out)
    y1 = oracle.compose_fwd(base, lora, g, s)
    y2 = oracle.compose_fwd_stable(base, lora, g, s)
    scale = np.abs(base) + s * np.abs(lora)
    assert np.max(np.abs(y1 - y2) / scale) < 1e-14


def test_compose_special_cases():
    rng = np.random.default_rng(7)
    base = rng.standard_normal((5, 6))
    lora = rng.standard_normal((5, 6))
    g = rng.uniform(0.5, 1.5, 6)
    # s = 0: the adapter drops out, y = g * base
    assert np.array_equal(oracle.compose_fwd(base, lora, g, 0.0), g * base)
    # lora = 0 and g = 1: identity on base
    assert np.array_equal(oracle.compose_fwd_stable(base, 0 * lora, np.ones(6), 0.9), base)


def _loss(dy, base, lora, m, n, s):
    return np.sum(dy * oracle.compose_fwd(base, lora, m / n, s))


def test_compose_bwd_central_differences():
    rng = np.random.default_rng(8)
    T, out, s = 9, 7, 1.1
    base = rng.standard_normal((T, out))
    lora = rng.standard_normal((T, out))
    dy = rng.standard_normal((T, out))
    n = rng.uniform(0.5, 2.0, out)
    m = rng.uniform(0.5, 2.0, out)
    db, dl, dm = oracle.compose_bwd(dy, base, lora, m / n, n, s)
    h = 1e-4   # L is linear in each argument: the central difference is exact up to rounding
    for j in range(out):
        e = np.zeros(out)
        e[j] = h
        fd = (_loss(dy, base, lora, m + e, n, s) - _loss(dy, base, lora, m - e, n, s)) / (2 * h)
        assert abs(fd - dm[j]) <= 1e-9 * max(1.0, abs(dm[j]))
    for (t, j) in [(0, 0), (3, 5), (8, 6), (4, 2)]:
        E = np.zeros((T, out))
        E[t, j] = h
        fdb = (_loss(dy, base + E, lora, m, n, s) - _loss(dy, base - E, lora, m, n, s)) / (2 * h)
        fdl = (_loss(dy, base, lora + E, m, n, s) - _loss(dy, base, lora - E, m, n, s)) / (2 * h)
        assert abs(fdb - db[t, j]) <= 1e-9 * max(1.0, abs(db[t, j]))
        assert abs(fdl - dl[t, j]) <= 1e-9 * max(1.0, abs(dl[t, j]))


def test_compose_bwd_homogeneity_identity():
    # y is linear in m for fixed n, so sum_j m_j d_mag_j = sum_{t,j} dy * y
    rng = np.random.default_rng(9)
    T, out, s = 33, 21, 0.6
    base = rng.standard_normal((T, out))
    lora = rng.standard_normal((T, out))
    dy = rng.standard_normal((T, out))
    n = rng.uniform(0.5, 2.0, out)
    m = rng.uniform(0.5, 2.0, out)
    _, _, dm = oracle.compose_bwd(dy, base, lora, m / n, n, s)
    lhs = np.sum(m * dm)
    rhs = np.sum(dy * oracle.compose_fwd(base, lora, m / n, s))
    assert abs(lhs - rhs) <= 1e-12 * np.sum(np.abs(dy) * (np.abs(base) + s * np.abs(lora)))


def test_naive_bf16_collapse_example():
    # g = 1 + 2^-8 rounds to exactly 1.0 in bf16 (a tie to even), so the naive
    # path returns base unchanged; the exact y = 3 * (1 + 2^-8) = 3.01171875
    # lies above the midpoint 3.0078125 and rounds to 3.015625 in bf16.
    base = np.array([[0x4040]], np.uint16)          # 3.0
    lora = np.array([[0x0000]], np.uint16)          # 0.0
    g = np.array([1 + 2 ** -8])
    naive = oracle.compose_fwd_naive_bf16(base, lora, g, 1.0)
    assert naive[0, 0] == 0x4040
    exact = oracle.compose_fwd_stable(oracle.bf16_bits_to_f64(base), 0.0 * oracle.bf16_bits_to_f64(lora), g, 1.0)
    assert exact[0, 0] == 3.01171875
    assert oracle.f64_to_bf16_bits(exact)[0, 0] == 0x4041   # 3.015625


def test_naive_bf16_matches_hand_steps():
    # base 1.5, lora 0.25, s = 3, g = 0.75 (all exact in bf16):
    # RN(3*0.25)=0.75, RN(1.5+0.75)=2.25, RN(0.75*2.25)=RN(1.6875)=1.6875
    base = np.array([[0x3FC0]], np.uint16)   # 1.5
    lora = np.array([[0x3E80]], np.uint16)   # 0.25
    got = oracle.compose_fwd_naive_bf16(base, lora, np.array([0.75]), 3.0)
    assert oracle.bf16_bits_to_f64(got)[0, 0] == 1.6875


# --------------------------------------------------------------------------
# gradient through the norm (the non-detached variant)
# --------------------------------------------------------------------------

def _norm_grad_case(seed, out=5, inp=7, r=3, s=0.9):
    rng = np.random.default_rng(seed)
    W0 = rng.standard_normal((out, inp)) / np.sqrt(inp)
    A = rng.standard_normal((r, inp)) / np.sqrt(inp)
    B = rng.standard_normal((out, r)) * 0.3
    m = rng.uniform(0.5, 1.5, out)
    w = rng.standard_normal(out)          # dL/dg
    return W0, A, B, m, w, s


def _g_loss(W0, A, B, m, w, s):
    # L(A, B) = <w, g(A, B)>, g = m / n through the (separately pinned) norm
    _, g = oracle.weight_norm(W0, A, B, m, s)
    return float(np.sum(w * g))


def _grad_inputs(W0, A, B, m, w, s):
    n, g = oracle.weight_norm(W0, A, B, m, s)
    return n, g, w / n                    # d_mag = dL/dm = (dL/dg) / n


def test_norm_grad_central_differences():
    W0, A, B, m, w, s = _norm_grad_case(21)
    n, g, d_mag = _grad_inputs(W0, A, B, m, w, s)
    dA, dB = oracle.norm_grad(W0, A, B, s, n, g, d_mag)
    assert dA.shape == A.shape and dB.shape == B.shape
    h = 1e-6
    for X, dX, which in ((A, dA, "A"), (B, dB, "B")):
        for idx in np.ndindex(X.shape):
            E = np.zeros_like(X)
            E[idx] = h
            if which == "A":
                fd = (_g_loss(W0, A + E, B, m, w, s) - _g_loss(W0, A - E, B, m, w, s)) / (2 * h)
            else:
                fd = (_g_loss(W0, A, B + E, m, w, s) - _g_loss(W0, A, B - E, m, w, s)) / (2 * h)
            assert abs(fd - dX[idx]) <= 1e-7 * max(1.0, abs(dX[idx])), (which, idx, fd, dX[idx])


def test_norm_grad_matches_torch_autograd_of_dense_definition():
    torch = pytest.importorskip("torch")
    W0, A, B, m, w, s = _norm_grad_case(22, out=9, inp=13, r=4, s=1.7)
    n, g, d_mag = _grad_inputs(W0, A, B, m, w, s)
    dA, dB = oracle.norm_grad(W0, A, B, s, n, g, d_mag)
    tA = torch.tensor(A, dtype=torch.float64, requires_grad=True)
    tB = torch.tensor(B, dtype=torch.float64, requires_grad=True)
    V = torch.tensor(W0, dtype=torch.float64) + s * (tB @ tA)
    L = torch.sum(torch.tensor(w * m) / torch.linalg.vector_norm(V, dim=1))
    gA, gB = torch.autograd.grad(L, (tA, tB))
    assert np.allclose(dA, gA.numpy(), rtol=1e-12, atol=1e-14)
    assert np.allclose(dB, gB.numpy(), rtol=1e-12, atol=1e-14)


def test_norm_grad_euler_identity_without_base():
    # W0 = 0: n_i = s ||B_i A|| is homogeneous of degree 1 in A and in B, so
    # <A, dA> = <B, dB> = sum_i (dL/dn_i) n_i with dL/dn = -g d_mag
    W0, A, B, m, w, s = _norm_grad_case(23, out=11, inp=17, r=5)
    W0 = np.zeros_like(W0)
    n, g, d_mag = _grad_inputs(W0, A, B, m, w, s)
    dA, dB = oracle.norm_grad(W0, A, B, s, n, g, d_mag)
    want = float(np.sum(-g * d_mag * n))
    scale = float(np.sum(np.abs(g * d_mag * n)))
    assert abs(np.sum(A * dA) - want) <= 1e-12 * scale
    assert abs(np.sum(B * dB) - want) <= 1e-12 * scale
    assert abs(want) > 1e-3 * scale


def test_norm_grad_b_zero_closed_form():
    # B = 0: V = W0, dA = s B^T dV = 0; with A = [I_r | 0], W0 A^T is the first
    # r columns of W0, so dB_i = s (dL/dn_i / n_i) W0[i, :r], n_i = ||W0_i||
    rng = np.random.default_rng(24)
    out, inp, r, s = 6, 10, 3, 1.3
    W0 = rng.standard_normal((out, inp))
    A = np.zeros((r, inp))
    A[np.arange(r), np.arange(r)] = 1.0
    B = np.zeros((out, r))
    m = rng.uniform(0.5, 1.5, out)
    d_mag = rng.standard_normal(out)
    n = np.linalg.norm(W0, axis=1)
    g = m / n
    dA, dB = oracle.norm_grad(W0, A, B, s, n, g, d_mag)
    assert np.array_equal(dA, np.zeros_like(A))
    want = s * (-g * d_mag / n)[:, None] * W0[:, :r]
    assert np.allclose(dB, want, rtol=1e-14, atol=0)


def test_norm_grad_row_and_column_subsets():
    # the sampled large-shape checks rely on these: dB rows need only their own
    # rows, dA columns only their own columns of W0 and A
    W0, A, B, m, w, s = _norm_grad_case(25, out=12, inp=16, r=4)
    n, g, d_mag = _grad_inputs(W0, A, B, m, w, s)
    dA, dB = oracle.norm_grad(W0, A, B, s, n, g, d_mag)
    rows = np.array([0, 5, 11])
    cols = np.array([1, 2, 15])
    _, dB_r = oracle.norm_grad(W0[rows], A, B[rows], s, n[rows], g[rows], d_mag[rows])
    dA_c, _ = oracle.norm_grad(W0[:, cols], A[:, cols], B, s, n, g, d_mag)
    assert np.allclose(dB_r, dB[rows], rtol=1e-13, atol=0)
    assert np.allclose(dA_c, dA[:, cols], rtol=1e-13, atol=0)


# --------------------------------------------------------------------------
# the compose with its adjacent products
# --------------------------------------------------------------------------

def test_layer_forward_one_hot_closed_form():
    # one-hot token rows pick single entries: base[t, j] = W0[j, k_t] and
    # lora[t, j] = B[j, q_t], so y[t, j] = g_j (W0[j, k_t] + s B[j, q_t])
    rng = np.random.default_rng(31)
    T, inp, out, r, s = 6, 9, 7, 4, 1.7
    W0 = rng.standard_normal((out, inp))
    B = rng.standard_normal((out, r))
    g = rng.uniform(0.5, 1.5, out)
    k = np.array([0, 3, 8, 3, 5, 1])
    q = np.array([2, 0, 3, 1, 1, 2])
    x = np.zeros((T, inp))
    x[np.arange(T), k] = 1.0
    xa = np.zeros((T, r))
    xa[np.arange(T), q] = 1.0
    want = g[None, :] * (W0[:, k].T + s * B[:, q].T)
    assert np.allclose(oracle.linear_fwd(x, W0, xa, B, g, s), want, rtol=1e-15, atol=0)
    base = rng.standard_normal((T, out))
    want_l = g[None, :] * (base + s * B[:, q].T)
    assert np.allclose(oracle.compose_lora_fwd(base, xa, B, g, s), want_l, rtol=1e-15, atol=0)

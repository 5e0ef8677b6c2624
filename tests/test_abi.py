"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, sizes workspaces, and rejects bad arguments before touching
the GPU.  CPU only (no compute call is made)."""
import os
import re

import pytest

import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import build as dbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    dbuild.build()
    return dora.load_library()


def _declared():
    names = set()
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", h)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(dora_\w+)\s*\(", txt))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "dora_norm_factored" in names and "dora_compose_fwd" in names and "dora_compose_bwd" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(9):
        s = dora.dora_status_str(code)
        assert s.startswith("DORA_")
    assert dora.dora_status_str(0) == "DORA_OK"


def test_norm_workspace_is_rank_dependent_only():
    d = 8192
    dense = d * d * 4       # one fp32 out x in matrix, 256 MiB
    prev = 0
    for r in (16, 64, 128, 256, 384, 512, 768):
        ws = dora.dora_norm_factored_workspace(d, d, r)
        assert 0 < ws < dense
        assert ws > prev
        prev = ws
        # O((out + in) r + r^2) with a bounded constant
        assert ws <= 24 * (2 * d * r + r * r) + (1 << 20)
    # doubling out at fixed r grows the workspace far less than out*in would
    assert dora.dora_norm_factored_workspace(2 * d, d, 64) < 2 * dora.dora_norm_factored_workspace(d, d, 64)


def test_bwd_workspace():
    assert dora.dora_compose_bwd_workspace(15360, 8192) >= 8192 * 4
    assert dora.dora_compose_bwd_workspace(15360, 8192) <= 256 * 8192 * 4
    assert dora.dora_compose_bwd_workspace(0, 8192) > 0
    assert dora.dora_compose_bwd_workspace(-1, 8) == 0


def test_invalid_shapes_give_zero_workspace():
    assert dora.dora_norm_factored_workspace(8, 0, 4) == 0
    assert dora.dora_norm_factored_workspace(8, 16, 0) == 0
    assert dora.dora_norm_factored_workspace(-1, 16, 4) == 0
    assert dora.dora_norm_factored_workspace(8, 16, 4096) == 0


FAKE = 1 << 20   # a 256-byte aligned non-null address: never dereferenced on these paths


def test_norm_argument_errors(lib):
    f = lib.dora_norm_factored
    ok = dict(W0=FAKE, A=FAKE, B=FAKE, m=FAKE, s=1.0, out=256, inp=64, r=8, norm=FAKE, g=FAKE, ws=FAKE,
              wsb=1 << 30, stream=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["W0"], a["A"], a["B"], a["m"], a["s"], a["out"], a["inp"], a["r"], a["norm"], a["g"],
                 a["ws"], a["wsb"], a["stream"])

    assert call(out=-1) == 2
    assert call(inp=0) == 2
    assert call(r=0) == 2
    assert call(r=2000) == 2
    assert call(out=0) == 0                     # empty: no-op
    assert call(W0=None) == 1
    assert call(g=None) == 1
    assert call(inp=66) == 3                    # row stride not a multiple of 16 bytes
    assert call(W0=FAKE + 4) == 3
    assert call(B=FAKE + 8) == 3
    assert call(ws=None) == 5
    assert call(ws=FAKE + 16) == 5
    assert call(wsb=16) == 5


def test_compose_argument_errors(lib):
    fwd = lib.dora_compose_fwd
    assert fwd(7, FAKE, FAKE, FAKE, 1.0, 4, 8, FAKE, None) == 4          # dtype
    assert fwd(1, FAKE, FAKE, FAKE, 1.0, -1, 8, FAKE, None) == 2
    assert fwd(1, FAKE, FAKE, FAKE, 1.0, 0, 8, FAKE, None) == 0          # empty
    assert fwd(1, FAKE, FAKE, FAKE, 1.0, 4, 0, FAKE, None) == 0
    assert fwd(1, None, FAKE, FAKE, 1.0, 4, 8, FAKE, None) == 1
    assert fwd(1, FAKE + 1, FAKE, FAKE, 1.0, 4, 8, FAKE, None) == 3     # bf16 element misaligned
    assert fwd(0, FAKE + 2, FAKE, FAKE, 1.0, 4, 8, FAKE, None) == 3     # f32 element misaligned
    bwd = lib.dora_compose_bwd
    args = [1, FAKE, FAKE, FAKE, FAKE, FAKE, 1.0, 64, 64, FAKE, FAKE, FAKE, FAKE, 1 << 30, None]

    def call(i, v):
        a = list(args)
        a[i] = v
        return bwd(*a)

    assert call(0, 9) == 4
    assert call(7, -2) == 2
    assert call(8, 0) == 0
    assert call(1, None) == 1
    assert call(11, None) == 1
    assert call(12, None) == 5
    assert call(12, FAKE + 64) == 5
    assert call(13, 4) == 5
    assert call(9, FAKE + 1) == 3


def test_launch_counter_starts_at_zero(lib):
    assert dora.dora_kernel_launches() >= 0


def test_bf16_norm_workspace_and_argument_errors(lib):
    d = 8192
    prev = 0
    for r in (16, 64, 128, 256, 384, 512, 768):
        ws = dora.dora_norm_factored_bf16_workspace(d, d, r)
        assert 0 < ws < d * d * 2          # never the size of a bf16 out x in matrix
        assert ws > prev
        prev = ws
    assert dora.dora_norm_factored_bf16_workspace(d, d, 0) == 0
    assert dora.dora_norm_factored_bf16_workspace(d, 0, 8) == 0
    f = lib.dora_norm_factored_bf16
    ok = dict(W0=FAKE, A=FAKE, B=FAKE, m=FAKE, n0=FAKE, s=1.0, out=256, inp=64, r=8, norm=FAKE, g=FAKE, ws=FAKE,
              wsb=1 << 30, stream=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["W0"], a["A"], a["B"], a["m"], a["n0"], a["s"], a["out"], a["inp"], a["r"], a["norm"], a["g"],
                 a["ws"], a["wsb"], a["stream"])

    assert call(out=-1) == 2
    assert call(r=0) == 2
    assert call(out=0) == 0
    assert call(n0=None) == 1
    assert call(W0=None) == 1
    assert call(inp=60) == 3                    # bf16 row stride not a multiple of 16 bytes
    assert call(A=FAKE + 8) == 3
    assert call(ws=FAKE + 16) == 5
    assert call(wsb=16) == 5
    rs = lib.dora_row_sumsq_bf16
    assert rs(FAKE, -1, 64, FAKE, None) == 2
    assert rs(FAKE, 0, 64, FAKE, None) == 0
    assert rs(None, 4, 64, FAKE, None) == 1
    assert rs(FAKE, 4, 60, FAKE, None) == 3
    assert rs(FAKE + 8, 4, 64, FAKE, None) == 3


def test_norm_bwd_workspace_and_argument_errors(lib):
    d = 8192
    prev = 0
    for r in (16, 64, 128, 256, 384, 512, 768):
        ws = dora.dora_norm_factored_bwd_workspace(d, d, r)
        assert 0 < ws < d * d * 4          # never the size of an fp32 out x in matrix
        assert ws > prev
        prev = ws
    assert dora.dora_norm_factored_bwd_workspace(d, d, 0) == 0
    assert dora.dora_norm_factored_bwd_workspace(d, 0, 8) == 0
    assert dora.dora_norm_factored_bwd_workspace(-1, 8, 8) == 0
    f = lib.dora_norm_factored_bwd
    ok = dict(W0=FAKE, A=FAKE, B=FAKE, n=FAKE, g=FAKE, dm=FAKE, s=1.0, out=256, inp=64, r=8, dA=FAKE, dB=FAKE,
              ws=FAKE, wsb=1 << 30, stream=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["W0"], a["A"], a["B"], a["n"], a["g"], a["dm"], a["s"], a["out"], a["inp"], a["r"], a["dA"],
                 a["dB"], a["ws"], a["wsb"], a["stream"])

    assert call(out=-1) == 2
    assert call(inp=0) == 2
    assert call(r=0) == 2
    assert call(r=2000) == 2
    assert call(out=0, dA=None) == 1             # out = 0 still writes dA (zeros)
    assert call(W0=None) == 1
    assert call(dm=None) == 1
    assert call(dB=None) == 1
    assert call(inp=66) == 3                    # row stride not a multiple of 16 bytes
    assert call(W0=FAKE + 4) == 3
    assert call(B=FAKE + 8) == 3
    assert call(dA=FAKE + 2) == 3
    assert call(ws=None) == 5
    assert call(ws=FAKE + 16) == 5
    assert call(wsb=16) == 5


def test_fused_forward_workspace_and_argument_errors(lib):
    assert dora.dora_compose_fused_workspace(8192, 384) >= 2 * 8192 * 384 * 2
    assert dora.dora_compose_fused_workspace(8192, 0) == 0
    assert dora.dora_compose_fused_workspace(-1, 8) == 0
    lf = lib.dora_compose_lora_fwd
    ok = dict(base=FAKE, xa=FAKE, B=FAKE, g=FAKE, s=1.0, T=64, out=256, r=16, y=FAKE, ws=FAKE, wsb=1 << 30,
              stream=None)

    def call(**kw):
        a = dict(ok, **kw)
        return lf(a["base"], a["xa"], a["B"], a["g"], a["s"], a["T"], a["out"], a["r"], a["y"], a["ws"], a["wsb"],
                  a["stream"])

    assert call(T=-1) == 2
    assert call(r=0) == 2
    assert call(T=0) == 0 and call(out=0) == 0           # empty: no-op
    assert call(base=None) == 1
    assert call(xa=None) == 1
    assert call(ws=None) == 5
    assert call(out=260) == 3                            # bf16 rows of 16 bytes
    assert call(r=12) == 3
    assert call(y=FAKE + 8) == 3
    assert call(base=FAKE + 2) == 3
    assert call(g=FAKE + 4) == 3                         # g is read 16 bytes at a time
    assert call(ws=FAKE + 16) == 5
    assert call(wsb=16) == 5
    lin = lib.dora_linear_fwd
    okl = dict(x=FAKE, W0=FAKE, xa=FAKE, B=FAKE, g=FAKE, s=1.0, T=64, inp=128, out=256, r=16, y=FAKE, ws=FAKE,
               wsb=1 << 30, stream=None)

    def call_l(**kw):
        a = dict(okl, **kw)
        return lin(a["x"], a["W0"], a["xa"], a["B"], a["g"], a["s"], a["T"], a["inp"], a["out"], a["r"], a["y"],
                   a["ws"], a["wsb"], a["stream"])

    assert call_l(inp=0) == 2
    assert call_l(T=0) == 0
    assert call_l(W0=None) == 1
    assert call_l(inp=12) == 3
    assert call_l(x=FAKE + 4) == 3
    assert call_l(wsb=16) == 5
    lb = lib.dora_compose_lora_fwd_bf16
    okb = dict(base=FAKE, xa=FAKE, B=FAKE, g=FAKE, s=1.0, T=64, out=256, r=16, y=FAKE, stream=None)

    def call_b(**kw):
        a = dict(okb, **kw)
        return lb(a["base"], a["xa"], a["B"], a["g"], a["s"], a["T"], a["out"], a["r"], a["y"], a["stream"])

    assert call_b(T=-1) == 2
    assert call_b(r=0) == 2
    assert call_b(T=0) == 0 and call_b(out=0) == 0       # empty: no-op
    assert call_b(B=None) == 1
    assert call_b(g=None) == 1
    assert call_b(out=260) == 3
    assert call_b(r=12) == 3
    assert call_b(B=FAKE + 8) == 3                       # bf16 B is a TMA operand: 16-byte aligned
    assert call_b(g=FAKE + 4) == 3

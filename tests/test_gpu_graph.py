"""The library's calls captured in a CUDA graph: after one call of each entry
point outside capture (which sets up the device and caches the plans and
tensor maps for those buffers), a training step captured with
torch.cuda.graph -- the factored norm, the compose forward and backward, the
norm gradient and both fused forms -- replays to the same bits as the same
calls launched one by one, on new input values written into the captured
buffers.  The eager results themselves are checked against the fp64 oracle by
the other parity tests; here they are also checked against the oracle once,
so that a replay that did nothing cannot pass."""
import pytest
import torch

import oracle
import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import DEV, act_to_dev, assert_no_device_error, check_rel, f32_dev, to_f64

pytestmark = pytest.mark.gpu


def _inputs(sh, seed):
    return wl.make_module(sh, seed)


def test_step_replays_bitwise_in_a_cuda_graph():
    sh = wl.shape("high_rank", T=512, inp=1024, out=1024, r=64)
    d0, d1 = _inputs(sh, 7101), _inputs(sh, 7102)
    s = d0["s"]
    W0, A, B, m = (f32_dev(d0[k]) for k in ("W0", "A", "B", "m"))
    base, lora, dy = (act_to_dev(d0[k]) for k in ("base", "lora", "dy"))
    xa = act_to_dev(d0["base"][:, : sh.r].copy())
    x = act_to_dev(d0["dy"][:, : sh.inp].copy())          # any bf16 [T, in] serves as x
    W0b = W0.to(torch.bfloat16)
    norm, g, dm = (torch.empty(sh.out, device=DEV) for _ in range(3))
    y, db, dl, yl, yx = (torch.empty_like(base) for _ in range(5))
    dA, dB = torch.empty_like(A), torch.empty_like(B)
    ws_n = torch.empty(dora.dora_norm_factored_workspace(sh.out, sh.inp, sh.r), dtype=torch.uint8, device=DEV)
    ws_b = torch.empty(dora.dora_compose_bwd_workspace(sh.T, sh.out), dtype=torch.uint8, device=DEV)
    ws_g = torch.empty(dora.dora_norm_factored_bwd_workspace(sh.out, sh.inp, sh.r), dtype=torch.uint8, device=DEV)
    ws_f = torch.empty(dora.dora_compose_fused_workspace(sh.out, sh.r), dtype=torch.uint8, device=DEV)
    outs = (norm, g, y, db, dl, dm, dA, dB, yl, yx)

    def step():
        st = torch.cuda.current_stream()
        dora.dora_norm_factored(W0, A, B, m, s, norm, g, ws_n, st)
        dora.dora_compose_fwd(base, lora, g, s, y, st)
        dora.dora_compose_bwd(dy, base, lora, g, norm, s, db, dl, dm, ws_b, st)
        dora.dora_norm_factored_bwd(W0, A, B, norm, g, dm, s, dA, dB, ws_g, st)
        dora.dora_compose_lora_fwd(base, xa, B, g, s, yl, ws_f, st)
        dora.dora_linear_fwd(x, W0b, xa, B, g, s, yx, ws_f, st)

    # one eager call of each (set-up and caches), then the reference results
    # for the second input set, computed eagerly
    step()
    torch.cuda.synchronize()

    def load(dd):
        for t, k in ((W0, "W0"), (A, "A"), (B, "B"), (m, "m")):
            t.copy_(f32_dev(dd[k]))
        for t, k in ((base, "base"), (lora, "lora"), (dy, "dy")):
            t.copy_(act_to_dev(dd[k]))
        xa.copy_(act_to_dev(dd["base"][:, : sh.r].copy()))
        x.copy_(act_to_dev(dd["dy"][:, : sh.inp].copy()))
        W0b.copy_(W0.to(torch.bfloat16))

    load(d1)
    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]
    # the eager norm is the oracle's (a replay that wrote nothing would keep
    # the first set's values, which the oracle check below also rejects)
    check_rel("eager norm", to_f64(eager[0]), oracle.adapted_row_norm(d1["W0"], d1["A"], d1["B"], s))

    load(d0)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    launches0 = dora.dora_kernel_launches()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    captured = dora.dora_kernel_launches() - launches0
    assert captured > 0

    for t in outs:
        t.fill_(float("nan"))
    load(d1)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert_no_device_error()
    # replays launch from the graph, not through the host entry points
    assert dora.dora_kernel_launches() - launches0 == captured
    names = ("norm", "g", "y", "d_base", "d_lora", "d_mag", "dA", "dB", "lora-form y", "linear-form y")
    for name, a, b in zip(names, outs, eager):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)), name

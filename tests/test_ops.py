"""torch.library registration of the hot path: the ops exist and their fake
(shape) implementations propagate shapes and dtypes without a GPU."""
import pytest

torch = pytest.importorskip("torch")


def test_ops_registered_and_fake_shapes():
    from torch._subclasses.fake_tensor import FakeTensorMode

    import parameter_efficient_fine_gb300.ops  # noqa: F401  (registers torch.ops.dora.*)

    for name in ("norm_factored", "row_sumsq", "norm_factored_bf16", "compose", "compose_bwd", "norm_factored_bwd",
                 "module"):
        assert hasattr(torch.ops.dora, name)
    with FakeTensorMode():
        W0 = torch.empty(64, 32, device="cuda")
        A = torch.empty(4, 32, device="cuda")
        B = torch.empty(64, 4, device="cuda")
        m = torch.empty(64, device="cuda")
        n, g = torch.ops.dora.norm_factored(W0, A, B, m, 1.0)
        assert n.shape == (64,) and g.shape == (64,) and n.dtype == torch.float32
        base = torch.empty(8, 64, device="cuda", dtype=torch.bfloat16)
        y = torch.ops.dora.compose(base, base, m, g, n, 1.0)
        assert y.shape == base.shape and y.dtype == torch.bfloat16
        db, dl, dm = torch.ops.dora.compose_bwd(base, base, base, g, n, 1.0)
        assert db.shape == base.shape and dl.dtype == torch.bfloat16 and dm.shape == (64,) and dm.dtype == torch.float32
        W16, A16, B16 = W0.bfloat16(), A.bfloat16(), B.bfloat16()
        n0 = torch.ops.dora.row_sumsq(W16)
        n16, g16 = torch.ops.dora.norm_factored_bf16(W16, A16, B16, m, n0, 1.0)
        assert n0.shape == (64,) and n0.dtype == torch.float32 and n16.shape == (64,) and g16.dtype == torch.float32
        dA, dB = torch.ops.dora.norm_factored_bwd(W0, A, B, n, g, m, 1.0)
        assert dA.shape == A.shape and dB.shape == B.shape and dA.dtype == torch.float32
        y2, n2, g2 = torch.ops.dora.module(base, base, W0, A, B, m, 1.0)
        assert y2.shape == base.shape and y2.dtype == torch.bfloat16 and n2.shape == (64,) and g2.shape == (64,)

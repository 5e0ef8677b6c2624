"""A seeded sweep of randomly drawn module shapes through the factored norm and
the compose forward and backward, each checked against the fp64 oracle under
the tolerances stated in gpu_util.py.  The hand-picked cases of the other
parity tests cover the tile edges their author thought of; these draw out, in,
r, T and the activation dtype from the ranges the library accepts, to reach
combinations nobody listed: compose grids whose rows do not divide the
resident blocks, norm N chunks and K tails of every size, single rows and
single tokens.  The shapes are fixed by the seed: the same on every run."""
import numpy as np
import pytest

from parameter_efficient_fine_gb300 import workloads as wl

from gpu_util import full_check

pytestmark = pytest.mark.gpu

N_SHAPES = 32


def drawn_shape(k: int):
    rng = np.random.default_rng(20261203 + k)
    out = int(rng.integers(1, 1601))
    inp = 4 * int(rng.integers(1, 401))          # the norm's TMA rows: in % 4 == 0
    r = int(rng.integers(1, 801))
    T = int(rng.integers(1, 701))
    act = "f32" if rng.random() < 0.25 else "bf16"
    return wl.shape("high_rank", out=out, inp=inp, r=r, T=T, act=act)


@pytest.mark.parametrize("k", range(N_SHAPES))
def test_drawn_shape(k):
    sh = drawn_shape(k)
    full_check(sh, 8800 + k)


def test_drawn_shapes_are_varied():
    # the draw reaches the cases it is for (checked on the host, no GPU work)
    shapes = [drawn_shape(k) for k in range(N_SHAPES)]
    assert any(s.act == "f32" for s in shapes) and any(s.act == "bf16" for s in shapes)
    assert any(s.r > 384 for s in shapes) and any(s.r <= 128 for s in shapes)
    assert any(s.out % 8 for s in shapes) and any(s.r % 4 for s in shapes)

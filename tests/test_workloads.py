"""Seeded input generator: determinism, shapes, distributions, bf16 rounding."""
import math

import numpy as np
import pytest

from parameter_efficient_fine_gb300 import workloads as wl


def test_tiny_shapes_and_determinism():
    sh = wl.shape("tiny")
    a = wl.make_module(sh, wl.seed_for("tiny"))
    b = wl.make_module(sh, wl.seed_for("tiny"))
    assert a["W0"].shape == (512, 512) and a["A"].shape == (16, 512) and a["B"].shape == (512, 16)
    assert a["base"].shape == (256, 512) and a["base"].dtype == np.float32
    for k in ("W0", "A", "B", "m", "base", "lora", "dy"):
        assert np.array_equal(a[k], b[k])
    assert a["s"] == 32 / 4
    c = wl.make_module(sh, wl.seed_for("tiny", 1))
    assert not np.array_equal(a["W0"], c["W0"])


def test_distributions_match_recipe():
    sh = wl.shape("high_rank", out=512, inp=2048, T=512)
    w = wl.make_weights(sh, 7)
    assert abs(w["W0"].std() - 1 / math.sqrt(2048)) < 0.02 / math.sqrt(2048) * 5
    assert abs(w["B"].std() - 0.01) < 0.001
    row = np.linalg.norm(w["W0"].astype(np.float64), axis=1)
    ratio = w["m"] / row - 1
    assert abs(ratio.std() - 1e-2) < 2e-3
    a = wl.make_activations(sh, 7)
    assert a["base"].dtype == np.uint16 and a["base"].shape == (512, 512)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(10000).astype(np.float32),
                        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, -0.0, 65504.0], np.float32)])
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(wl.f32_to_bf16_bits(x), want)

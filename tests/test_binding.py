"""The Python binding's failure modes, on the CPU: no library means an error
(never a CPU fallback), and host tensors are refused before any call reaches
the library (every pointer of the C ABI is a device pointer)."""
import os
import subprocess
import sys

import pytest
import torch

import parameter_efficient_fine_gb300 as dora
from parameter_efficient_fine_gb300 import build as dbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_missing_library_is_an_error():
    code = ("import parameter_efficient_fine_gb300 as d\n"
            "d._LIB_PATH = '/nonexistent/libdora.so'\n"
            "d._lib = None\n"
            "d.dora_norm_factored_workspace(8, 8, 1)\n")
    res = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode != 0
    assert "not built" in res.stderr


def test_host_tensors_are_refused():
    dbuild.build()
    W0, A, B, m = torch.zeros(8, 8), torch.zeros(1, 8), torch.zeros(8, 1), torch.ones(8)
    norm, g = torch.empty(8), torch.empty(8)
    ws = torch.empty(max(dora.dora_norm_factored_workspace(8, 8, 1), 1), dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensors"):
        dora.dora_norm_factored(W0, A, B, m, 1.0, norm, g, ws, stream=0)
    base = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensors"):
        dora.dora_compose_fwd(base, base, g, 1.0, torch.empty_like(base), stream=0)

"""DoRA weight-norm and compose hot path for GB300 (sm_103a).

Thin ctypes binding over libdora.so (include/dora.h).  Every function here only
marshals arguments -- shapes from tensor sizes, raw device pointers, the
current torch stream -- and calls the C entry point of the same name; all
arithmetic runs in the library's CUDA kernels.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os

__all__ = [
    "DoraError",
    "load_library",
    "library_path",
    "dora_status_str",
    "dora_norm_factored_workspace",
    "dora_norm_factored",
    "dora_row_sumsq_bf16",
    "dora_norm_factored_bf16_workspace",
    "dora_norm_factored_bf16",
    "dora_norm_factored_bwd_workspace",
    "dora_norm_factored_bwd",
    "dora_compose_fwd",
    "dora_compose_fused_workspace",
    "dora_compose_lora_fwd",
    "dora_compose_lora_fwd_bf16",
    "dora_linear_fwd",
    "dora_compose_bwd_workspace",
    "dora_compose_bwd",
    "dora_compose_bwd_noalloc",
    "dora_device_error",
    "dora_kernel_launches",
    "dora_test_stall_loads",
    "dora_test_fused_pairs",
    "DORA_F32",
    "DORA_BF16",
]

DORA_F32 = 0
DORA_BF16 = 1

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libdora.so")
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_sz = ctypes.c_size_t
_f32 = ctypes.c_float
_int = ctypes.c_int

_SIGNATURES = {
    "dora_status_str": (ctypes.c_char_p, [_int]),
    "dora_norm_factored_workspace": (_sz, [_i64, _i64, _i64]),
    "dora_norm_factored": (_int, [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _vp, _vp, _vp, _sz, _vp]),
    "dora_row_sumsq_bf16": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "dora_norm_factored_bf16_workspace": (_sz, [_i64, _i64, _i64]),
    "dora_norm_factored_bf16": (_int, [_vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _vp, _vp, _vp, _sz, _vp]),
    "dora_norm_factored_bwd_workspace": (_sz, [_i64, _i64, _i64]),
    "dora_norm_factored_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _vp, _vp, _vp, _sz, _vp]),
    "dora_compose_fwd": (_int, [_int, _vp, _vp, _vp, _f32, _i64, _i64, _vp, _vp]),
    "dora_compose_fused_workspace": (_sz, [_i64, _i64]),
    "dora_compose_lora_fwd": (_int, [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _vp, _vp, _sz, _vp]),
    "dora_compose_lora_fwd_bf16": (_int, [_vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _vp, _vp]),
    "dora_linear_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _i64, _i64, _vp, _vp, _sz, _vp]),
    "dora_compose_bwd_workspace": (_sz, [_i64, _i64]),
    "dora_compose_bwd": (_int, [_int, _vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "dora_compose_bwd_noalloc": (_int, [_int, _vp, _vp, _vp, _vp, _vp, _f32, _i64, _i64, _vp, _vp, _vp, _vp]),
    "dora_device_error": (_int, [ctypes.POINTER(_int)]),
    "dora_kernel_launches": (ctypes.c_uint64, []),
    "dora_test_stall_loads": (_int, [_int, ctypes.c_uint64]),
    "dora_test_fused_pairs": (_int, [_int]),
}


class DoraError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {load_library().dora_status_str(status).decode()}")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libdora.so (built by __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"libdora.so not built ({_LIB_PATH}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    # every pointer of the C ABI is a device pointer: a host tensor would hand
    # a host address to the kernels
    if not getattr(x, "is_cuda", False):
        raise ValueError(f"libdora takes CUDA tensors (device memory); got one on {getattr(x, 'device', type(x))}")
    return x.data_ptr()


def _stream(stream) -> int:
    if stream is not None:
        return stream if isinstance(stream, int) else stream.cuda_stream
    import torch
    return torch.cuda.current_stream().cuda_stream


def _act(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return DORA_F32
    if t.dtype == torch.bfloat16:
        return DORA_BF16
    raise TypeError(f"activation dtype {t.dtype} not supported (float32 or bfloat16)")


def _check(name: str, st: int) -> None:
    if st != 0:
        raise DoraError(name, st)


def dora_status_str(status: int) -> str:
    return load_library().dora_status_str(status).decode()


def dora_norm_factored_workspace(out: int, inp: int, r: int) -> int:
    return int(load_library().dora_norm_factored_workspace(out, inp, r))


def dora_compose_bwd_workspace(T: int, out: int) -> int:
    return int(load_library().dora_compose_bwd_workspace(T, out))


def dora_norm_factored(W0, A, B, m, s: float, norm, g, workspace, stream=None) -> None:
    """norm[i] = ||W0_i + s (B A)_i||, g = m / norm (see include/dora.h)."""
    out, inp = W0.shape
    r = A.shape[0]
    st = load_library().dora_norm_factored(
        _ptr(W0), _ptr(A), _ptr(B), _ptr(m), float(s), out, inp, r, _ptr(norm), _ptr(g),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("dora_norm_factored", st)


def dora_row_sumsq_bf16(W0, n0sq, stream=None) -> None:
    """n0sq[i] = sum_j W0[i, j]^2 for a bfloat16 W0 (see include/dora.h)."""
    rows, cols = W0.shape
    _check("dora_row_sumsq_bf16",
           load_library().dora_row_sumsq_bf16(_ptr(W0), rows, cols, _ptr(n0sq), _stream(stream)))


def dora_norm_factored_bf16_workspace(out: int, inp: int, r: int) -> int:
    return int(load_library().dora_norm_factored_bf16_workspace(out, inp, r))


def dora_norm_factored_bf16(W0, A, B, m, n0sq, s: float, norm, g, workspace, stream=None) -> None:
    """dora_norm_factored for bfloat16 W0, A, B with the base term from n0sq (see include/dora.h)."""
    out, inp = W0.shape
    r = A.shape[0]
    st = load_library().dora_norm_factored_bf16(
        _ptr(W0), _ptr(A), _ptr(B), _ptr(m), _ptr(n0sq), float(s), out, inp, r, _ptr(norm), _ptr(g),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("dora_norm_factored_bf16", st)


def dora_norm_factored_bwd_workspace(out: int, inp: int, r: int) -> int:
    return int(load_library().dora_norm_factored_bwd_workspace(out, inp, r))


def dora_norm_factored_bwd(W0, A, B, norm, g, d_mag, s: float, dA, dB, workspace, stream=None) -> None:
    """dA, dB: the gradient that flows through the row norm (see include/dora.h)."""
    out, inp = W0.shape
    r = A.shape[0]
    st = load_library().dora_norm_factored_bwd(
        _ptr(W0), _ptr(A), _ptr(B), _ptr(norm), _ptr(g), _ptr(d_mag), float(s), out, inp, r, _ptr(dA), _ptr(dB),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("dora_norm_factored_bwd", st)


def dora_compose_fwd(base, lora, g, s: float, y, stream=None) -> None:
    """y = base + (g-1)*base + g*s*lora (see include/dora.h)."""
    T, out = base.shape
    st = load_library().dora_compose_fwd(_act(base), _ptr(base), _ptr(lora), _ptr(g), float(s), T, out,
                                         _ptr(y), _stream(stream))
    _check("dora_compose_fwd", st)


def dora_compose_fused_workspace(out: int, r: int) -> int:
    return int(load_library().dora_compose_fused_workspace(out, r))


def dora_compose_lora_fwd(base, xa, B, g, s: float, y, workspace, stream=None) -> None:
    """y = base + (g-1) base + g s (xa B^T), lora formed in the kernel (see include/dora.h)."""
    T, out = base.shape
    r = xa.shape[1]
    st = load_library().dora_compose_lora_fwd(
        _ptr(base), _ptr(xa), _ptr(B), _ptr(g), float(s), T, out, r, _ptr(y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("dora_compose_lora_fwd", st)


def dora_compose_lora_fwd_bf16(base, xa, B, g, s: float, y, stream=None) -> None:
    """y = base + (g-1) base + g s (xa B^T) for a bf16 B: one product, s applied to
    the accumulator (see include/dora.h)."""
    T, out = base.shape
    r = xa.shape[1]
    st = load_library().dora_compose_lora_fwd_bf16(
        _ptr(base), _ptr(xa), _ptr(B), _ptr(g), float(s), T, out, r, _ptr(y), _stream(stream))
    _check("dora_compose_lora_fwd_bf16", st)


def dora_linear_fwd(x, W0, xa, B, g, s: float, y, workspace, stream=None) -> None:
    """y = g (x W0^T + s xa B^T) as one GEMM with the compose in its epilogue (see include/dora.h)."""
    T, inp = x.shape
    out = W0.shape[0]
    r = xa.shape[1]
    st = load_library().dora_linear_fwd(
        _ptr(x), _ptr(W0), _ptr(xa), _ptr(B), _ptr(g), float(s), T, inp, out, r, _ptr(y),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _check("dora_linear_fwd", st)


def dora_compose_bwd(grad_out, base, lora, g, norm, s: float, d_base, d_lora, d_mag, workspace,
                     stream=None) -> None:
    """d_base = g*dy, d_lora = s*g*dy, d_mag = sum_t dy*(base+s*lora)/norm (see include/dora.h)."""
    T, out = grad_out.shape
    st = load_library().dora_compose_bwd(
        _act(grad_out), _ptr(grad_out), _ptr(base), _ptr(lora), _ptr(g), _ptr(norm), float(s), T, out,
        _ptr(d_base), _ptr(d_lora), _ptr(d_mag), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check("dora_compose_bwd", st)


def dora_compose_bwd_noalloc(grad_out, base, lora, g, norm, s: float, d_base, d_lora, d_mag,
                             stream=None) -> None:
    """dora_compose_bwd without a workspace, for callers that cannot allocate
    device memory where they run the backward: the partial sums use the
    library's fixed device scratch array (see include/dora.h; calls that
    overlap on the GPU race on that array)."""
    T, out = grad_out.shape
    st = load_library().dora_compose_bwd_noalloc(
        _act(grad_out), _ptr(grad_out), _ptr(base), _ptr(lora), _ptr(g), _ptr(norm), float(s), T, out,
        _ptr(d_base), _ptr(d_lora), _ptr(d_mag), _stream(stream))
    _check("dora_compose_bwd_noalloc", st)


def dora_device_error() -> int:
    """Reads and clears the device error word (synchronises the device)."""
    code = _int(0)
    st = load_library().dora_device_error(ctypes.byref(code))
    if st not in (0, 8):
        raise DoraError("dora_device_error", st)
    return int(code.value)


def dora_kernel_launches() -> int:
    return int(load_library().dora_kernel_launches())


def dora_test_stall_loads(on: bool, wait_limit_ns: int = 0) -> None:
    """Testing hook: make later norm calls' bounded waits expire (see include/dora.h)."""
    _check("dora_test_stall_loads", load_library().dora_test_stall_loads(1 if on else 0, int(wait_limit_ns)))


def dora_test_fused_pairs(allow: bool) -> None:
    """Testing hook: run the fused kernels as single CTAs when False (see include/dora.h)."""
    _check("dora_test_fused_pairs", load_library().dora_test_fused_pairs(1 if allow else 0))

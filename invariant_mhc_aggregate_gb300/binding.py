"""Python binding of the C ABI in ``include/mhc_h_aggregate.h`` (ctypes).

Argument marshalling only: every step of the operation runs in the sm_103a
kernels of ``libmhc_h_aggregate.so``.  There is no CPU or PyTorch fallback; if
the library has not been built, loading it raises.

The function names match the C entry points.  Tensor arguments must be CUDA
tensors, contiguous, with the dtypes and shapes of the header; T and H are
read from ``residual``.  Calls are asynchronous on ``stream`` (default: the
current PyTorch stream of the tensors' device).
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

MHC_OK = 0
MHC_ERR_INVALID_ARG = 1
MHC_ERR_UNSUPPORTED = 2
MHC_ERR_CUDA = 3

MHC_PATH_NONE = -1
MHC_PATH_VEC16 = 0
MHC_PATH_PAIR = 1
MHC_PATH_ELEMENT = 2
MHC_PATH_VEC32 = 3
MHC_PATH_SHIFT16 = 4
PATH_NAMES = {MHC_PATH_NONE: "none", MHC_PATH_VEC16: "vec16", MHC_PATH_PAIR: "pair",
              MHC_PATH_ELEMENT: "element", MHC_PATH_VEC32: "vec32", MHC_PATH_SHIFT16: "shift16"}

MHC_DTYPE_BF16 = 0
MHC_DTYPE_F16 = 1

#: Every symbol the header declares, in declaration order.
EXPORTS = (
    "mhc_h_aggregate_abi_version",
    "mhc_h_aggregate_fwd",
    "mhc_h_aggregate_bwd",
    "mhc_h_aggregate_fwd_path",
    "mhc_h_aggregate_bwd_path",
    "mhc_aggregate_fwd",
    "mhc_aggregate_bwd",
    "mhc_aggregate_fwd_path",
    "mhc_aggregate_bwd_path",
    "mhc_pre_sigmoid",
    "mhc_aggregate_sigmoid_fwd",
    "mhc_aggregate_sigmoid_bwd",
    "mhc_sigmoid_param_grad",
    "mhc_post_fwd",
    "mhc_post_bwd",
    "mhc_post_sigmoid_fwd",
    "mhc_post_sigmoid_bwd",
    "mhc_post_fwd_path",
    "mhc_post_bwd_path",
    "mhc_status_string",
    "mhc_h_aggregate_last_cuda_error",
    "mhc_h_aggregate_wait_timeouts",
)

_lock = threading.Lock()
_lib = None


class MhcError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        lib = load()
        text = lib.mhc_status_string(status).decode()
        if status == MHC_ERR_CUDA:
            text += f" (cudaError {lib.mhc_h_aggregate_last_cuda_error()})"
        super().__init__(f"{what}: {text}")


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load the compiled library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        path = path or _build.LIB_PATH
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        i32 = ctypes.c_int32
        lib.mhc_h_aggregate_abi_version.argtypes = []
        lib.mhc_h_aggregate_abi_version.restype = i32
        lib.mhc_h_aggregate_fwd.argtypes = [p, p, p, i64, i64, p]
        lib.mhc_h_aggregate_fwd.restype = i32
        lib.mhc_h_aggregate_bwd.argtypes = [p, p, p, p, p, i64, i64, p]
        lib.mhc_h_aggregate_bwd.restype = i32
        lib.mhc_h_aggregate_fwd_path.argtypes = [p, p, p, i64, i64]
        lib.mhc_h_aggregate_fwd_path.restype = i32
        lib.mhc_h_aggregate_bwd_path.argtypes = [p, p, p, p, p, i64, i64]
        lib.mhc_h_aggregate_bwd_path.restype = i32
        lib.mhc_aggregate_fwd.argtypes = [p, p, p, i64, i32, i64, i32, p]
        lib.mhc_aggregate_fwd.restype = i32
        lib.mhc_aggregate_bwd.argtypes = [p, p, p, p, p, i64, i32, i64, i32, p]
        lib.mhc_aggregate_bwd.restype = i32
        lib.mhc_aggregate_fwd_path.argtypes = [p, p, p, i64, i32, i64]
        lib.mhc_aggregate_fwd_path.restype = i32
        lib.mhc_aggregate_bwd_path.argtypes = [p, p, p, p, p, i64, i32, i64]
        lib.mhc_aggregate_bwd_path.restype = i32
        lib.mhc_pre_sigmoid.argtypes = [p, p, p, p, i64, i32, p]
        lib.mhc_pre_sigmoid.restype = i32
        lib.mhc_aggregate_sigmoid_fwd.argtypes = [p, p, p, p, p, i64, i32, i64, i32, p]
        lib.mhc_aggregate_sigmoid_fwd.restype = i32
        lib.mhc_aggregate_sigmoid_bwd.argtypes = [p, p, p, p, p, p, p, p, i64, i32, i64, i32, p]
        lib.mhc_aggregate_sigmoid_bwd.restype = i32
        lib.mhc_sigmoid_param_grad.argtypes = [p, p, p, p, i64, i32, p]
        lib.mhc_sigmoid_param_grad.restype = i32
        lib.mhc_post_fwd.argtypes = [p, p, p, p, p, i64, i32, i64, i32, p]
        lib.mhc_post_fwd.restype = i32
        lib.mhc_post_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i64, i32, i64, i32, p]
        lib.mhc_post_bwd.restype = i32
        lib.mhc_post_sigmoid_fwd.argtypes = [p, p, p, p, p, p, p, i64, i32, i64, i32, p]
        lib.mhc_post_sigmoid_fwd.restype = i32
        lib.mhc_post_sigmoid_bwd.argtypes = [p, p, p, p, p, p, p, p, p, p, p, p, i64, i32, i64, i32, p]
        lib.mhc_post_sigmoid_bwd.restype = i32
        lib.mhc_post_fwd_path.argtypes = [p, p, p, p, p, i64, i32, i64]
        lib.mhc_post_fwd_path.restype = i32
        lib.mhc_post_bwd_path.argtypes = [p, p, p, p, p, p, p, p, p, i64, i32, i64]
        lib.mhc_post_bwd_path.restype = i32
        lib.mhc_status_string.argtypes = [i32]
        lib.mhc_status_string.restype = ctypes.c_char_p
        lib.mhc_h_aggregate_last_cuda_error.argtypes = []
        lib.mhc_h_aggregate_last_cuda_error.restype = i32
        lib.mhc_h_aggregate_wait_timeouts.argtypes = []
        lib.mhc_h_aggregate_wait_timeouts.restype = i64
        if path == _build.LIB_PATH:
            _lib = lib
        return lib


# ---------------------------------------------------------------------------
# raw entry points: integer addresses, sizes and a stream handle
# ---------------------------------------------------------------------------

def fwd_raw(residual: int, pre: int, out: int, T: int, H: int, stream: int = 0) -> int:
    return load().mhc_h_aggregate_fwd(residual, pre, out, T, H, stream)


def bwd_raw(grad_out: int, residual: int, pre: int, grad_residual: int, grad_pre: int,
            T: int, H: int, stream: int = 0) -> int:
    return load().mhc_h_aggregate_bwd(grad_out, residual, pre, grad_residual, grad_pre, T, H,
                                      stream)


def fwd_path_raw(residual: int, pre: int, out: int, T: int, H: int) -> int:
    return load().mhc_h_aggregate_fwd_path(residual, pre, out, T, H)


def bwd_path_raw(grad_out: int, residual: int, pre: int, grad_residual: int, grad_pre: int,
                 T: int, H: int) -> int:
    return load().mhc_h_aggregate_bwd_path(grad_out, residual, pre, grad_residual, grad_pre, T, H)


def agg_fwd_raw(residual: int, pre: int, out: int, T: int, n: int, H: int, dtype: int,
                stream: int = 0) -> int:
    return load().mhc_aggregate_fwd(residual, pre, out, T, n, H, dtype, stream)


def agg_bwd_raw(grad_out: int, residual: int, pre: int, grad_residual: int, grad_pre: int,
                T: int, n: int, H: int, dtype: int, stream: int = 0) -> int:
    return load().mhc_aggregate_bwd(grad_out, residual, pre, grad_residual, grad_pre, T, n, H,
                                    dtype, stream)


def agg_fwd_path_raw(residual: int, pre: int, out: int, T: int, n: int, H: int) -> int:
    return load().mhc_aggregate_fwd_path(residual, pre, out, T, n, H)


def agg_bwd_path_raw(grad_out: int, residual: int, pre: int, grad_residual: int, grad_pre: int,
                     T: int, n: int, H: int) -> int:
    return load().mhc_aggregate_bwd_path(grad_out, residual, pre, grad_residual, grad_pre, T, n, H)


def pre_sigmoid_raw(mix: int, alpha: int, b: int, pre: int, T: int, n: int, stream: int = 0) -> int:
    return load().mhc_pre_sigmoid(mix, alpha, b, pre, T, n, stream)


def agg_sigmoid_fwd_raw(residual: int, mix: int, alpha: int, b: int, out: int, T: int, n: int,
                        H: int, dtype: int, stream: int = 0) -> int:
    return load().mhc_aggregate_sigmoid_fwd(residual, mix, alpha, b, out, T, n, H, dtype, stream)


def agg_sigmoid_bwd_raw(grad_out: int, residual: int, mix: int, alpha: int, b: int,
                        grad_residual: int, grad_z: int, grad_mix: int, T: int, n: int, H: int,
                        dtype: int, stream: int = 0) -> int:
    return load().mhc_aggregate_sigmoid_bwd(grad_out, residual, mix, alpha, b, grad_residual,
                                            grad_z, grad_mix, T, n, H, dtype, stream)


def sigmoid_param_grad_raw(grad_z: int, mix: int, grad_b: int, grad_alpha: int, T: int, n: int,
                           stream: int = 0) -> int:
    return load().mhc_sigmoid_param_grad(grad_z, mix, grad_b, grad_alpha, T, n, stream)


def wait_timeouts() -> int:
    """1 if a bounded wait of the bulk-copy kernels ran out on the current
    device since the last call, else 0 (clears it; synchronizes the device);
    -1 on a CUDA error."""
    return int(load().mhc_h_aggregate_wait_timeouts())


def post_fwd_raw(x: int, y: int, post: int, res: int, out: int, T: int, n: int, H: int, dtype: int,
                 stream: int = 0) -> int:
    return load().mhc_post_fwd(x, y, post, res, out, T, n, H, dtype, stream)


def post_bwd_raw(grad_out: int, x: int, y: int, post: int, res: int, grad_x: int, grad_y: int,
                 grad_post: int, grad_res: int, T: int, n: int, H: int, dtype: int,
                 stream: int = 0) -> int:
    return load().mhc_post_bwd(grad_out, x, y, post, res, grad_x, grad_y, grad_post, grad_res,
                               T, n, H, dtype, stream)


def post_sigmoid_fwd_raw(x: int, y: int, mix: int, alpha: int, b: int, res: int, out: int, T: int, n: int,
                         H: int, dtype: int, stream: int = 0) -> int:
    return load().mhc_post_sigmoid_fwd(x, y, mix, alpha, b, res, out, T, n, H, dtype, stream)


def post_sigmoid_bwd_raw(grad_out: int, x: int, y: int, mix: int, alpha: int, b: int, res: int,
                         grad_x: int, grad_y: int, grad_z: int, grad_mix: int, grad_res: int, T: int,
                         n: int, H: int, dtype: int, stream: int = 0) -> int:
    return load().mhc_post_sigmoid_bwd(grad_out, x, y, mix, alpha, b, res, grad_x, grad_y, grad_z,
                                       grad_mix, grad_res, T, n, H, dtype, stream)


def post_fwd_path_raw(x: int, y: int, post: int, res: int, out: int, T: int, n: int, H: int) -> int:
    return load().mhc_post_fwd_path(x, y, post, res, out, T, n, H)


def post_bwd_path_raw(grad_out: int, x: int, y: int, post: int, res: int, grad_x: int, grad_y: int,
                      grad_post: int, grad_res: int, T: int, n: int, H: int) -> int:
    return load().mhc_post_bwd_path(grad_out, x, y, post, res, grad_x, grad_y, grad_post,
                                    grad_res, T, n, H)


# ---------------------------------------------------------------------------
# tensor entry points
# ---------------------------------------------------------------------------

_TORCH_DTYPES = {torch.bfloat16: MHC_DTYPE_BF16, torch.float16: MHC_DTYPE_F16}

def _check(t: torch.Tensor, name: str, dtype, shape):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor, got {t.device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_handle(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return int(stream.cuda_stream)
    return int(stream)


def _TH(residual: torch.Tensor) -> tuple[int, int]:
    if residual.dim() != 3 or residual.shape[1] != 4:
        raise ValueError(f"residual must be [T,4,H], got {tuple(residual.shape)}")
    return int(residual.shape[0]), int(residual.shape[2])


def mhc_h_aggregate_fwd(residual: torch.Tensor, pre: torch.Tensor, out: torch.Tensor,
                        stream=None) -> None:
    """out[t,h] = bf16((pre0*r0 + pre1*r1) + (pre2*r2 + pre3*r3)), written into ``out``."""
    T, H = _TH(residual)
    _check(residual, "residual", torch.bfloat16, (T, 4, H))
    _check(pre, "pre", torch.float32, (T, 4))
    _check(out, "out", torch.bfloat16, (T, H))
    st = fwd_raw(residual.data_ptr(), pre.data_ptr(), out.data_ptr(), T, H,
                 _stream_handle(stream, residual.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_h_aggregate_fwd")


def mhc_h_aggregate_bwd(grad_out: torch.Tensor, residual: torch.Tensor, pre: torch.Tensor,
                        grad_residual: torch.Tensor, grad_pre: torch.Tensor,
                        stream=None) -> None:
    """grad_residual = bf16(pre*g), grad_pre = ORDER-256 sums of g*r; written in place."""
    T, H = _TH(residual)
    _check(grad_out, "grad_out", torch.bfloat16, (T, H))
    _check(residual, "residual", torch.bfloat16, (T, 4, H))
    _check(pre, "pre", torch.float32, (T, 4))
    _check(grad_residual, "grad_residual", torch.bfloat16, (T, 4, H))
    _check(grad_pre, "grad_pre", torch.float32, (T, 4))
    st = bwd_raw(grad_out.data_ptr(), residual.data_ptr(), pre.data_ptr(),
                 grad_residual.data_ptr(), grad_pre.data_ptr(), T, H,
                 _stream_handle(stream, residual.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_h_aggregate_bwd")


def mhc_h_aggregate_fwd_path(residual: torch.Tensor, pre: torch.Tensor, out: torch.Tensor) -> int:
    T, H = _TH(residual)
    return fwd_path_raw(residual.data_ptr(), pre.data_ptr(), out.data_ptr(), T, H)


def mhc_h_aggregate_bwd_path(grad_out, residual, pre, grad_residual, grad_pre) -> int:
    T, H = _TH(residual)
    return bwd_path_raw(grad_out.data_ptr(), residual.data_ptr(), pre.data_ptr(),
                        grad_residual.data_ptr(), grad_pre.data_ptr(), T, H)


def _TnH(residual: torch.Tensor) -> tuple[int, int, int]:
    if residual.dim() != 3:
        raise ValueError(f"residual must be [T,n,H], got {tuple(residual.shape)}")
    return int(residual.shape[0]), int(residual.shape[1]), int(residual.shape[2])


def _storage(t: torch.Tensor, name: str) -> int:
    if t.dtype not in _TORCH_DTYPES:
        raise TypeError(f"{name} must be bfloat16 or float16, got {t.dtype}")
    return _TORCH_DTYPES[t.dtype]


def mhc_aggregate_fwd(residual: torch.Tensor, pre: torch.Tensor, out: torch.Tensor,
                      stream=None) -> None:
    """General forward: residual [T,n,H] (bf16 or f16), pre [T,n] fp32 -> out [T,H]."""
    T, n, H = _TnH(residual)
    dt = _storage(residual, "residual")
    _check(residual, "residual", residual.dtype, (T, n, H))
    _check(pre, "pre", torch.float32, (T, n))
    _check(out, "out", residual.dtype, (T, H))
    st = agg_fwd_raw(residual.data_ptr(), pre.data_ptr(), out.data_ptr(), T, n, H, dt,
                     _stream_handle(stream, residual.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_aggregate_fwd")


def mhc_aggregate_bwd(grad_out: torch.Tensor, residual: torch.Tensor, pre: torch.Tensor,
                      grad_residual: torch.Tensor, grad_pre: torch.Tensor, stream=None) -> None:
    """General backward for n streams and bf16 / f16 storage, written in place."""
    T, n, H = _TnH(residual)
    dt = _storage(residual, "residual")
    _check(grad_out, "grad_out", residual.dtype, (T, H))
    _check(residual, "residual", residual.dtype, (T, n, H))
    _check(pre, "pre", torch.float32, (T, n))
    _check(grad_residual, "grad_residual", residual.dtype, (T, n, H))
    _check(grad_pre, "grad_pre", torch.float32, (T, n))
    st = agg_bwd_raw(grad_out.data_ptr(), residual.data_ptr(), pre.data_ptr(),
                     grad_residual.data_ptr(), grad_pre.data_ptr(), T, n, H, dt,
                     _stream_handle(stream, residual.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_aggregate_bwd")


def aggregate(residual: torch.Tensor, pre: torch.Tensor, stream=None) -> torch.Tensor:
    """Allocate ``out`` [T,H] and run the general forward."""
    T, n, H = _TnH(residual)
    out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    mhc_aggregate_fwd(residual, pre, out, stream)
    return out


def aggregate_backward(grad_out: torch.Tensor, residual: torch.Tensor, pre: torch.Tensor,
                       stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Allocate and return (grad_residual [T,n,H], grad_pre [T,n] fp32)."""
    T, n, H = _TnH(residual)
    grad_residual = torch.empty((T, n, H), dtype=residual.dtype, device=residual.device)
    grad_pre = torch.empty((T, n), dtype=torch.float32, device=residual.device)
    mhc_aggregate_bwd(grad_out, residual, pre, grad_residual, grad_pre, stream)
    return grad_residual, grad_pre


def h_aggregate(residual: torch.Tensor, pre: torch.Tensor, stream=None) -> torch.Tensor:
    """Allocate ``out`` [T,H] BF16 and run the forward."""
    T, H = _TH(residual)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=residual.device)
    mhc_h_aggregate_fwd(residual, pre, out, stream)
    return out


def h_aggregate_backward(grad_out: torch.Tensor, residual: torch.Tensor, pre: torch.Tensor,
                         stream=None) -> tuple[torch.Tensor, torch.Tensor]:
    """Allocate and return (grad_residual [T,4,H] BF16, grad_pre [T,4] FP32)."""
    T, H = _TH(residual)
    grad_residual = torch.empty((T, 4, H), dtype=torch.bfloat16, device=residual.device)
    grad_pre = torch.empty((T, 4), dtype=torch.float32, device=residual.device)
    mhc_h_aggregate_bwd(grad_out, residual, pre, grad_residual, grad_pre, stream)
    return grad_residual, grad_pre


# ---------------------------------------------------------------------------
# the pre coefficients computed from the mix: pre = sigmoid(alpha * mix + b)
# ---------------------------------------------------------------------------

def _coeff_params(alpha: torch.Tensor, b: torch.Tensor, n: int, device) -> None:
    _check(b, "b", torch.float32, (n,))
    if not isinstance(alpha, torch.Tensor) or alpha.numel() != 1:
        raise ValueError("alpha must be a one-element tensor")
    _check(alpha, "alpha", torch.float32, tuple(alpha.shape))
    if alpha.device != device or b.device != device:
        raise ValueError("alpha and b must be on the device of the other tensors")


def mhc_pre_sigmoid(mix: torch.Tensor, alpha: torch.Tensor, b: torch.Tensor, pre: torch.Tensor,
                    stream=None) -> None:
    """pre[t,k] = sigmoid(alpha * mix[t,k] + b[k]) (the library's binary32 sigmoid)."""
    if mix.dim() != 2:
        raise ValueError(f"mix must be [T,n], got {tuple(mix.shape)}")
    T, n = int(mix.shape[0]), int(mix.shape[1])
    _check(mix, "mix", torch.float32, (T, n))
    _check(pre, "pre", torch.float32, (T, n))
    _coeff_params(alpha, b, n, mix.device)
    st = pre_sigmoid_raw(mix.data_ptr(), alpha.data_ptr(), b.data_ptr(), pre.data_ptr(), T, n,
                         _stream_handle(stream, mix.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_pre_sigmoid")


def mhc_aggregate_sigmoid_fwd(residual: torch.Tensor, mix: torch.Tensor, alpha: torch.Tensor,
                              b: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """out = aggregate(residual, sigmoid(alpha * mix + b)) in one kernel."""
    T, n, H = _TnH(residual)
    dt = _storage(residual, "residual")
    _check(residual, "residual", residual.dtype, (T, n, H))
    _check(mix, "mix", torch.float32, (T, n))
    _check(out, "out", residual.dtype, (T, H))
    _coeff_params(alpha, b, n, residual.device)
    st = agg_sigmoid_fwd_raw(residual.data_ptr(), mix.data_ptr(), alpha.data_ptr(), b.data_ptr(),
                             out.data_ptr(), T, n, H, dt, _stream_handle(stream, residual.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_aggregate_sigmoid_fwd")


def mhc_aggregate_sigmoid_bwd(grad_out: torch.Tensor, residual: torch.Tensor, mix: torch.Tensor,
                              alpha: torch.Tensor, b: torch.Tensor, grad_residual: torch.Tensor,
                              grad_z: torch.Tensor, grad_mix: torch.Tensor, stream=None) -> None:
    """Fused backward: grad_residual, grad_z = grad_pre * sigmoid'(z), grad_mix = alpha * grad_z."""
    T, n, H = _TnH(residual)
    dt = _storage(residual, "residual")
    _check(grad_out, "grad_out", residual.dtype, (T, H))
    _check(residual, "residual", residual.dtype, (T, n, H))
    _check(mix, "mix", torch.float32, (T, n))
    _check(grad_residual, "grad_residual", residual.dtype, (T, n, H))
    _check(grad_z, "grad_z", torch.float32, (T, n))
    _check(grad_mix, "grad_mix", torch.float32, (T, n))
    _coeff_params(alpha, b, n, residual.device)
    st = agg_sigmoid_bwd_raw(grad_out.data_ptr(), residual.data_ptr(), mix.data_ptr(),
                             alpha.data_ptr(), b.data_ptr(), grad_residual.data_ptr(),
                             grad_z.data_ptr(), grad_mix.data_ptr(), T, n, H, dt,
                             _stream_handle(stream, residual.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_aggregate_sigmoid_bwd")


def mhc_sigmoid_param_grad(grad_z: torch.Tensor, mix: torch.Tensor, grad_b: torch.Tensor,
                           grad_alpha: torch.Tensor, stream=None) -> None:
    """grad_b [n] and grad_alpha [1]: sums over tokens in ORDER-256."""
    if grad_z.dim() != 2:
        raise ValueError(f"grad_z must be [T,n], got {tuple(grad_z.shape)}")
    T, n = int(grad_z.shape[0]), int(grad_z.shape[1])
    _check(grad_z, "grad_z", torch.float32, (T, n))
    _check(mix, "mix", torch.float32, (T, n))
    _check(grad_b, "grad_b", torch.float32, (n,))
    if grad_alpha.numel() != 1:
        raise ValueError("grad_alpha must be a one-element tensor")
    _check(grad_alpha, "grad_alpha", torch.float32, tuple(grad_alpha.shape))
    st = sigmoid_param_grad_raw(grad_z.data_ptr(), mix.data_ptr(), grad_b.data_ptr(),
                                grad_alpha.data_ptr(), T, n, _stream_handle(stream, grad_z.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_sigmoid_param_grad")


def pre_sigmoid(mix: torch.Tensor, alpha: torch.Tensor, b: torch.Tensor, stream=None) -> torch.Tensor:
    pre = torch.empty_like(mix)
    mhc_pre_sigmoid(mix, alpha, b, pre, stream)
    return pre


def aggregate_sigmoid(residual: torch.Tensor, mix: torch.Tensor, alpha: torch.Tensor,
                      b: torch.Tensor, stream=None) -> torch.Tensor:
    """Allocate ``out`` [T,H] and run the fused forward."""
    T, n, H = _TnH(residual)
    out = torch.empty((T, H), dtype=residual.dtype, device=residual.device)
    mhc_aggregate_sigmoid_fwd(residual, mix, alpha, b, out, stream)
    return out


def aggregate_sigmoid_backward(grad_out: torch.Tensor, residual: torch.Tensor, mix: torch.Tensor,
                               alpha: torch.Tensor, b: torch.Tensor, stream=None):
    """Allocate and return (grad_residual [T,n,H], grad_z [T,n], grad_mix [T,n])."""
    T, n, H = _TnH(residual)
    grad_residual = torch.empty((T, n, H), dtype=residual.dtype, device=residual.device)
    grad_z = torch.empty((T, n), dtype=torch.float32, device=residual.device)
    grad_mix = torch.empty((T, n), dtype=torch.float32, device=residual.device)
    mhc_aggregate_sigmoid_bwd(grad_out, residual, mix, alpha, b, grad_residual, grad_z, grad_mix,
                              stream)
    return grad_residual, grad_z, grad_mix


def sigmoid_param_grad(grad_z: torch.Tensor, mix: torch.Tensor, stream=None):
    """Allocate and return (grad_b [n], grad_alpha [1])."""
    n = int(grad_z.shape[1])
    grad_b = torch.empty((n,), dtype=torch.float32, device=grad_z.device)
    grad_alpha = torch.empty((1,), dtype=torch.float32, device=grad_z.device)
    mhc_sigmoid_param_grad(grad_z, mix, grad_b, grad_alpha, stream)
    return grad_b, grad_alpha


# ---------------------------------------------------------------------------
# mHC post: out[t,k] = tree_n(res[t,k,j] * x[t,j]) + post[t,k] * y[t]
# ---------------------------------------------------------------------------

def _post_shapes(x: torch.Tensor, y: torch.Tensor, post: torch.Tensor, res: torch.Tensor):
    T, n, H = _TnH(x)
    dt = _storage(x, "x")
    _check(x, "x", x.dtype, (T, n, H))
    _check(y, "y", x.dtype, (T, H))
    _check(post, "post", torch.float32, (T, n))
    _check(res, "res", torch.float32, (T, n, n))
    return T, n, H, dt


def mhc_post_fwd(x: torch.Tensor, y: torch.Tensor, post: torch.Tensor, res: torch.Tensor,
                 out: torch.Tensor, stream=None) -> None:
    """out [T,n,H] = the n streams mixed by res plus post times the layer output y."""
    T, n, H, dt = _post_shapes(x, y, post, res)
    _check(out, "out", x.dtype, (T, n, H))
    st = post_fwd_raw(x.data_ptr(), y.data_ptr(), post.data_ptr(), res.data_ptr(), out.data_ptr(),
                      T, n, H, dt, _stream_handle(stream, x.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_post_fwd")


def mhc_post_bwd(grad_out: torch.Tensor, x: torch.Tensor, y: torch.Tensor, post: torch.Tensor,
                 res: torch.Tensor, grad_x: torch.Tensor, grad_y: torch.Tensor,
                 grad_post: torch.Tensor, grad_res: torch.Tensor, stream=None) -> None:
    """Fused backward: grad_x, grad_y, and grad_post / grad_res summed over H in ORDER-256."""
    T, n, H, dt = _post_shapes(x, y, post, res)
    _check(grad_out, "grad_out", x.dtype, (T, n, H))
    _check(grad_x, "grad_x", x.dtype, (T, n, H))
    _check(grad_y, "grad_y", x.dtype, (T, H))
    _check(grad_post, "grad_post", torch.float32, (T, n))
    _check(grad_res, "grad_res", torch.float32, (T, n, n))
    st = post_bwd_raw(grad_out.data_ptr(), x.data_ptr(), y.data_ptr(), post.data_ptr(),
                      res.data_ptr(), grad_x.data_ptr(), grad_y.data_ptr(), grad_post.data_ptr(),
                      grad_res.data_ptr(), T, n, H, dt, _stream_handle(stream, x.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_post_bwd")


def post(x: torch.Tensor, y: torch.Tensor, post_coeffs: torch.Tensor, res: torch.Tensor,
         stream=None) -> torch.Tensor:
    """Allocate ``out`` [T,n,H] and run the post forward."""
    out = torch.empty_like(x)
    mhc_post_fwd(x, y, post_coeffs, res, out, stream)
    return out


def post_backward(grad_out: torch.Tensor, x: torch.Tensor, y: torch.Tensor,
                  post_coeffs: torch.Tensor, res: torch.Tensor, stream=None):
    """Allocate and return (grad_x [T,n,H], grad_y [T,H], grad_post [T,n], grad_res [T,n,n])."""
    T, n, H = _TnH(x)
    grad_x = torch.empty_like(x)
    grad_y = torch.empty((T, H), dtype=x.dtype, device=x.device)
    grad_post = torch.empty((T, n), dtype=torch.float32, device=x.device)
    grad_res = torch.empty((T, n, n), dtype=torch.float32, device=x.device)
    mhc_post_bwd(grad_out, x, y, post_coeffs, res, grad_x, grad_y, grad_post, grad_res, stream)
    return grad_x, grad_y, grad_post, grad_res


# ---------------------------------------------------------------------------
# mHC post with post = sigmoid(alpha * mix + b) computed in the kernels
# ---------------------------------------------------------------------------

def mhc_post_sigmoid_fwd(x: torch.Tensor, y: torch.Tensor, mix: torch.Tensor, alpha: torch.Tensor,
                         b: torch.Tensor, res: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """out = the mHC post with post = sigmoid(alpha * mix + b), in one kernel."""
    T, n, H, dt = _post_shapes(x, y, mix, res)
    _check(out, "out", x.dtype, (T, n, H))
    _coeff_params(alpha, b, n, x.device)
    st = post_sigmoid_fwd_raw(x.data_ptr(), y.data_ptr(), mix.data_ptr(), alpha.data_ptr(), b.data_ptr(),
                              res.data_ptr(), out.data_ptr(), T, n, H, dt, _stream_handle(stream, x.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_post_sigmoid_fwd")


def mhc_post_sigmoid_bwd(grad_out: torch.Tensor, x: torch.Tensor, y: torch.Tensor, mix: torch.Tensor,
                         alpha: torch.Tensor, b: torch.Tensor, res: torch.Tensor, grad_x: torch.Tensor,
                         grad_y: torch.Tensor, grad_z: torch.Tensor, grad_mix: torch.Tensor,
                         grad_res: torch.Tensor, stream=None) -> None:
    """Fused backward: grad_x, grad_y, grad_res, and grad_z = grad_post * sigmoid'(z),
    grad_mix = alpha * grad_z in the epilogue."""
    T, n, H, dt = _post_shapes(x, y, mix, res)
    _check(grad_out, "grad_out", x.dtype, (T, n, H))
    _check(grad_x, "grad_x", x.dtype, (T, n, H))
    _check(grad_y, "grad_y", x.dtype, (T, H))
    _check(grad_z, "grad_z", torch.float32, (T, n))
    _check(grad_mix, "grad_mix", torch.float32, (T, n))
    _check(grad_res, "grad_res", torch.float32, (T, n, n))
    _coeff_params(alpha, b, n, x.device)
    st = post_sigmoid_bwd_raw(grad_out.data_ptr(), x.data_ptr(), y.data_ptr(), mix.data_ptr(),
                              alpha.data_ptr(), b.data_ptr(), res.data_ptr(), grad_x.data_ptr(),
                              grad_y.data_ptr(), grad_z.data_ptr(), grad_mix.data_ptr(), grad_res.data_ptr(),
                              T, n, H, dt, _stream_handle(stream, x.device))
    if st != MHC_OK:
        raise MhcError(st, "mhc_post_sigmoid_bwd")


def post_sigmoid(x: torch.Tensor, y: torch.Tensor, mix: torch.Tensor, alpha: torch.Tensor,
                 b: torch.Tensor, res: torch.Tensor, stream=None) -> torch.Tensor:
    """Allocate ``out`` [T,n,H] and run the post with post from the mix."""
    out = torch.empty_like(x)
    mhc_post_sigmoid_fwd(x, y, mix, alpha, b, res, out, stream)
    return out


def post_sigmoid_backward(grad_out: torch.Tensor, x: torch.Tensor, y: torch.Tensor, mix: torch.Tensor,
                          alpha: torch.Tensor, b: torch.Tensor, res: torch.Tensor, stream=None):
    """Allocate and return (grad_x [T,n,H], grad_y [T,H], grad_z [T,n], grad_mix [T,n],
    grad_res [T,n,n])."""
    T, n, H = _TnH(x)
    grad_x = torch.empty_like(x)
    grad_y = torch.empty((T, H), dtype=x.dtype, device=x.device)
    grad_z = torch.empty((T, n), dtype=torch.float32, device=x.device)
    grad_mix = torch.empty((T, n), dtype=torch.float32, device=x.device)
    grad_res = torch.empty((T, n, n), dtype=torch.float32, device=x.device)
    mhc_post_sigmoid_bwd(grad_out, x, y, mix, alpha, b, res, grad_x, grad_y, grad_z, grad_mix, grad_res,
                         stream)
    return grad_x, grad_y, grad_z, grad_mix, grad_res

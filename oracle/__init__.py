"""CPU oracle for the batch-invariant mHC pre "H Aggregate" (forward and backward).

TEST INFRASTRUCTURE ONLY.  The arithmetic lives in ``mhc_oracle.c`` (plain C11,
``-O2 -ffp-contract=off``, no fast math); this module compiles it with the host
``gcc`` and marshals numpy arrays through ``ctypes``.  Only the tests, the
package smoke check and the benchmark's CPU-baseline leg may import it; the
product path never does.  It shares no code with the CUDA library.

BF16 data is carried as ``numpy.uint16`` bit patterns.  Shapes follow the
"Add batch-invariant h_aggregate kernel" page (Summary): residual ``[T,4,H]``
BF16, pre ``[T,4]`` FP32, out ``[T,H]`` BF16; the backward adds g ``[T,H]``
BF16, grad_residual ``[T,4,H]`` BF16 and grad_pre ``[T,4]`` FP32.

Parity status of each function (what pins it, from the oracle pin tests):
  * bf16_from_float / float_from_bf16: exhaustive round trip, hand tie cases,
    agreement with torch's CPU conversion.
  * fwd: hand-worked examples (tree order, no FMA), exact-rational emulation,
    FP64 error bound, one-hot / zero / symmetry / scaling invariants.
  * grad_residual: hand-worked double-rounding examples, exact-rational
    emulation, identity and one-hot invariants.
  * grad_pre: integer-valued exact sums, FP64 error bound, hand-worked sparse
    cases that fix every level of the ORDER-256 tree.
  * f16_from_float / float_from_f16: exhaustive round trip, hand ties and
    edges, agreement with torch's CPU conversion.
  * aggregate_fwd / aggregate_bwd (stream count n in {1,2,4,8}, BF16 or FP16
    storage; a reading beyond the pages): hand-worked tree-order cases for n = 2
    and 8, equality with fwd/bwd at n = 4 BF16, exact-rational emulation,
    integer-valued exact sums, one-hot invariants.
  * exp32 / sigmoid32 (the fixed binary32 sequence that defines the sigmoid of
    the fused pre coefficients): hand-worked values, exact-rational emulation of
    every step, error bounds against FP64 e^x and sigmoid on a dense sample,
    exact special values, symmetry and monotonicity.
  * pre_sigmoid / aggregate_sigmoid_fwd / aggregate_sigmoid_bwd /
    sigmoid_param_grad (the "perf: fuse mHC coefficient backward epilogue"
    page's pre coefficients, a reading): FP64 bounds, exact special cases
    (z = 0, integer-valued sums), hand-worked token-order cases and an
    independent recursive builder of ORDER-256 over tokens.
  * post_fwd / post_bwd (mHC post, a reading not on the pages): hand-worked
    tree-order cases, exact-rational emulation, identity and zero special
    cases, integer-valued exact sums for grad_res and grad_post, FP64 bounds.
  * post_sigmoid_fwd / post_sigmoid_bwd (post coefficients from their own
    mix, a reading): z = 0 makes post = 0.5 and grad_z = grad_post / 4
    exactly (exact-rational forward, integer-valued grad_post); the
    pre-activation and epilogue wiring against numpy binary32 arithmetic on
    the pinned sigmoid and post.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmhc_oracle.so")

#: Compiler flags.  ``-ffp-contract=off`` stops GCC from fusing a multiply and
#: an add into an FMA (GCC's default on aarch64); ISO C11 mode also keeps the
#: GNU extensions that relax float semantics off.
CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-Wall", "-Wextra", "-Werror"]

_lock = threading.Lock()
_default = None


def library_path() -> str:
    return _LIB_PATH


def compile_library(src: str, out: str, extra_flags=()) -> str:
    """Compile an oracle C source into a shared library at ``out`` (atomic replace)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    try:
        subprocess.run(["gcc", *CFLAGS, *extra_flags, "-o", tmp, src], check=True,
                       capture_output=True, text=True)
        os.replace(tmp, out)
    except subprocess.CalledProcessError as e:
        raise RuntimeError(f"oracle build failed:\n{e.stderr}") from e
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle shared library if it is missing or older than its source."""
    with _lock:
        stale = (not os.path.exists(_LIB_PATH)
                 or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
        if force or stale:
            compile_library(_SRC, _LIB_PATH)
    return _LIB_PATH


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _shape_TH(residual: np.ndarray) -> tuple[int, int]:
    if residual.ndim != 3 or residual.shape[1] != 4:
        raise ValueError(f"residual must be [T,4,H], got {residual.shape}")
    return int(residual.shape[0]), int(residual.shape[2])


_DTYPES = {"bf16": 0, "f16": 1}


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_float_from_bf16.argtypes = [ctypes.c_uint16]
        lib.oracle_float_from_bf16.restype = ctypes.c_float
        lib.oracle_bf16_from_float.argtypes = [ctypes.c_float]
        lib.oracle_bf16_from_float.restype = ctypes.c_uint16
        for name in ("oracle_bf16_from_float_array", "oracle_float_from_bf16_array"):
            getattr(lib, name).argtypes = [p, p, i64]
            getattr(lib, name).restype = None
        lib.oracle_h_aggregate_fwd.argtypes = [p, p, p, i64, i64]
        lib.oracle_h_aggregate_fwd.restype = None
        lib.oracle_h_aggregate_bwd_grad_residual.argtypes = [p, p, p, i64, i64]
        lib.oracle_h_aggregate_bwd_grad_residual.restype = None
        lib.oracle_h_aggregate_bwd_grad_pre.argtypes = [p, p, p, i64, i64]
        lib.oracle_h_aggregate_bwd_grad_pre.restype = None
        lib.oracle_h_aggregate_bwd.argtypes = [p, p, p, p, p, i64, i64]
        lib.oracle_h_aggregate_bwd.restype = None
        for name in ("oracle_f16_from_float_array", "oracle_float_from_f16_array"):
            getattr(lib, name).argtypes = [p, p, i64]
            getattr(lib, name).restype = None
        lib.oracle_aggregate_fwd.argtypes = [p, p, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_aggregate_fwd.restype = ctypes.c_int
        lib.oracle_aggregate_bwd.argtypes = [p, p, p, p, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_aggregate_bwd.restype = ctypes.c_int
        lib.oracle_exp32_array.argtypes = [p, p, i64]
        lib.oracle_exp32_array.restype = None
        lib.oracle_sigmoid32_array.argtypes = [p, p, p, i64]
        lib.oracle_sigmoid32_array.restype = None
        lib.oracle_pre_sigmoid.argtypes = [p, p, p, p, i64, i64]
        lib.oracle_pre_sigmoid.restype = ctypes.c_int
        lib.oracle_aggregate_sigmoid_fwd.argtypes = [p, p, p, p, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_aggregate_sigmoid_fwd.restype = ctypes.c_int
        lib.oracle_aggregate_sigmoid_bwd.argtypes = [p, p, p, p, p, p, p, p, i64, i64, i64,
                                                     ctypes.c_int]
        lib.oracle_aggregate_sigmoid_bwd.restype = ctypes.c_int
        lib.oracle_sigmoid_param_grad.argtypes = [p, p, p, p, i64, i64]
        lib.oracle_sigmoid_param_grad.restype = ctypes.c_int
        lib.oracle_post_fwd.argtypes = [p, p, p, p, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_post_fwd.restype = ctypes.c_int
        lib.oracle_post_bwd.argtypes = [p, p, p, p, p, p, p, p, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_post_bwd.restype = ctypes.c_int
        lib.oracle_post_sigmoid_fwd.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, ctypes.c_int]
        lib.oracle_post_sigmoid_fwd.restype = ctypes.c_int
        lib.oracle_post_sigmoid_bwd.argtypes = [p, p, p, p, p, p, p, p, p, p, p, p, i64, i64, i64,
                                                ctypes.c_int]
        lib.oracle_post_sigmoid_bwd.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def bf16_from_float(self, x) -> np.ndarray:
        """Round float32 values to BF16 (RNE); returns uint16 patterns."""
        x = _as(x, np.float32)
        y = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_bf16_from_float_array(_ptr(x), _ptr(y), x.size)
        return y

    def float_from_bf16(self, x) -> np.ndarray:
        """Widen BF16 patterns (uint16) to float32 exactly."""
        x = _as(x, np.uint16)
        y = np.empty(x.shape, dtype=np.float32)
        self.lib.oracle_float_from_bf16_array(_ptr(x), _ptr(y), x.size)
        return y

    def f16_from_float(self, x) -> np.ndarray:
        """Round float32 values to IEEE binary16 (RNE); returns uint16 patterns."""
        x = _as(x, np.float32)
        y = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f16_from_float_array(_ptr(x), _ptr(y), x.size)
        return y

    def float_from_f16(self, x) -> np.ndarray:
        """Widen IEEE binary16 patterns (uint16) to float32 exactly."""
        x = _as(x, np.uint16)
        y = np.empty(x.shape, dtype=np.float32)
        self.lib.oracle_float_from_f16_array(_ptr(x), _ptr(y), x.size)
        return y

    def aggregate_fwd(self, residual, pre, dtype: str = "bf16") -> np.ndarray:
        """General stream count n (residual [T,n,H], pre [T,n]) and storage dtype
        ("bf16" or "f16"): out = cvt(balanced pairwise tree of pre_k * r_k)."""
        residual = _as(residual, np.uint16)
        pre = _as(pre, np.float32)
        T, n, H = residual.shape
        if pre.shape != (T, n):
            raise ValueError(f"pre must be [{T},{n}], got {pre.shape}")
        out = np.empty((T, H), dtype=np.uint16)
        if self.lib.oracle_aggregate_fwd(_ptr(residual), _ptr(pre), _ptr(out), T, n, H,
                                         _DTYPES[dtype]) != 0:
            raise ValueError(f"unsupported n={n} or dtype={dtype}")
        return out

    def aggregate_bwd(self, g, residual, pre, dtype: str = "bf16") -> tuple[np.ndarray, np.ndarray]:
        """(grad_residual uint16 [T,n,H], grad_pre float32 [T,n]) for stream count n."""
        g = _as(g, np.uint16)
        residual = _as(residual, np.uint16)
        pre = _as(pre, np.float32)
        T, n, H = residual.shape
        if g.shape != (T, H) or pre.shape != (T, n):
            raise ValueError("shape mismatch between g, residual and pre")
        gr = np.empty((T, n, H), dtype=np.uint16)
        gp = np.empty((T, n), dtype=np.float32)
        if self.lib.oracle_aggregate_bwd(_ptr(g), _ptr(residual), _ptr(pre), _ptr(gr), _ptr(gp),
                                         T, n, H, _DTYPES[dtype]) != 0:
            raise ValueError(f"unsupported n={n} or dtype={dtype}")
        return gr, gp

    # -- the pre coefficients from the mix (sigmoid), fused into the aggregate --

    def exp32(self, x) -> np.ndarray:
        """The library's binary32 e^x (Cody-Waite reduction, degree-7 Taylor)."""
        x = _as(x, np.float32)
        y = np.empty(x.shape, dtype=np.float32)
        self.lib.oracle_exp32_array(_ptr(x), _ptr(y), x.size)
        return y

    def sigmoid32(self, z) -> tuple[np.ndarray, np.ndarray]:
        """(sigmoid(z), sigmoid'(z)) as defined by the binary32 sequence."""
        z = _as(z, np.float32)
        s = np.empty(z.shape, dtype=np.float32)
        ds = np.empty(z.shape, dtype=np.float32)
        self.lib.oracle_sigmoid32_array(_ptr(z), _ptr(s), _ptr(ds), z.size)
        return s, ds

    @staticmethod
    def _coeffs(mix, alpha, b):
        mix = _as(mix, np.float32)
        alpha = _as(np.asarray(alpha, dtype=np.float32).reshape(1), np.float32)
        b = _as(b, np.float32)
        if mix.ndim != 2 or b.shape != (mix.shape[1],):
            raise ValueError(f"mix must be [T,n] and b [n], got {mix.shape} and {b.shape}")
        return mix, alpha, b

    def pre_sigmoid(self, mix, alpha, b) -> np.ndarray:
        """pre[t,k] = sigmoid(alpha * mix[t,k] + b[k]); float32 [T,n]."""
        mix, alpha, b = self._coeffs(mix, alpha, b)
        T, n = mix.shape
        pre = np.empty((T, n), dtype=np.float32)
        if self.lib.oracle_pre_sigmoid(_ptr(mix), _ptr(alpha), _ptr(b), _ptr(pre), T, n) != 0:
            raise ValueError(f"unsupported n={n}")
        return pre

    def aggregate_sigmoid_fwd(self, residual, mix, alpha, b, dtype: str = "bf16") -> np.ndarray:
        """out = aggregate(residual, sigmoid(alpha * mix + b)); uint16 [T,H]."""
        residual = _as(residual, np.uint16)
        mix, alpha, b = self._coeffs(mix, alpha, b)
        T, n, H = residual.shape
        if mix.shape != (T, n):
            raise ValueError(f"mix must be [{T},{n}], got {mix.shape}")
        out = np.empty((T, H), dtype=np.uint16)
        if self.lib.oracle_aggregate_sigmoid_fwd(_ptr(residual), _ptr(mix), _ptr(alpha), _ptr(b),
                                                 _ptr(out), T, n, H, _DTYPES[dtype]) != 0:
            raise ValueError(f"unsupported n={n} or dtype={dtype}")
        return out

    def aggregate_sigmoid_bwd(self, g, residual, mix, alpha, b, dtype: str = "bf16"):
        """(grad_residual uint16 [T,n,H], grad_z float32 [T,n], grad_mix float32 [T,n])."""
        g = _as(g, np.uint16)
        residual = _as(residual, np.uint16)
        mix, alpha, b = self._coeffs(mix, alpha, b)
        T, n, H = residual.shape
        if g.shape != (T, H) or mix.shape != (T, n):
            raise ValueError("shape mismatch between g, residual and mix")
        gr = np.empty((T, n, H), dtype=np.uint16)
        gz = np.empty((T, n), dtype=np.float32)
        gm = np.empty((T, n), dtype=np.float32)
        if self.lib.oracle_aggregate_sigmoid_bwd(_ptr(g), _ptr(residual), _ptr(mix), _ptr(alpha),
                                                 _ptr(b), _ptr(gr), _ptr(gz), _ptr(gm), T, n, H,
                                                 _DTYPES[dtype]) != 0:
            raise ValueError(f"unsupported n={n} or dtype={dtype}")
        return gr, gz, gm

    def sigmoid_param_grad(self, grad_z, mix) -> tuple[np.ndarray, np.float32]:
        """(grad_b float32 [n], grad_alpha float32): sums over tokens in ORDER-256."""
        grad_z = _as(grad_z, np.float32)
        mix = _as(mix, np.float32)
        if grad_z.ndim != 2 or grad_z.shape != mix.shape:
            raise ValueError("grad_z and mix must both be [T,n]")
        T, n = grad_z.shape
        gb = np.empty(n, dtype=np.float32)
        ga = np.empty(1, dtype=np.float32)
        if self.lib.oracle_sigmoid_param_grad(_ptr(grad_z), _ptr(mix), _ptr(gb), _ptr(ga), T, n) != 0:
            raise ValueError(f"unsupported n={n}")
        return gb, ga[0]

    # -- mHC post (a reading: the layer output expanded onto the n streams) --

    @staticmethod
    def _post_args(x, y, post, res):
        x = _as(x, np.uint16)
        y = _as(y, np.uint16)
        post = _as(post, np.float32)
        res = _as(res, np.float32)
        T, n, H = x.shape
        if y.shape != (T, H) or post.shape != (T, n) or res.shape != (T, n, n):
            raise ValueError("shapes: x [T,n,H], y [T,H], post [T,n], res [T,n,n]")
        return x, y, post, res, T, n, H

    def post_fwd(self, x, y, post, res, dtype: str = "bf16") -> np.ndarray:
        """out[t,k,h] = cvt(tree_n(res[t,k,j] * x[t,j,h]) + post[t,k] * y[t,h]); [T,n,H]."""
        x, y, post, res, T, n, H = self._post_args(x, y, post, res)
        out = np.empty((T, n, H), dtype=np.uint16)
        if self.lib.oracle_post_fwd(_ptr(x), _ptr(y), _ptr(post), _ptr(res), _ptr(out), T, n, H,
                                    _DTYPES[dtype]) != 0:
            raise ValueError(f"unsupported n={n} or dtype={dtype}")
        return out

    def post_bwd(self, g, x, y, post, res, dtype: str = "bf16"):
        """(grad_x [T,n,H], grad_y [T,H], grad_post float32 [T,n], grad_res float32 [T,n,n])."""
        x, y, post, res, T, n, H = self._post_args(x, y, post, res)
        g = _as(g, np.uint16)
        if g.shape != (T, n, H):
            raise ValueError(f"g must be [{T},{n},{H}]")
        gx = np.empty((T, n, H), dtype=np.uint16)
        gy = np.empty((T, H), dtype=np.uint16)
        gp = np.empty((T, n), dtype=np.float32)
        gr = np.empty((T, n, n), dtype=np.float32)
        if self.lib.oracle_post_bwd(_ptr(g), _ptr(x), _ptr(y), _ptr(post), _ptr(res), _ptr(gx),
                                    _ptr(gy), _ptr(gp), _ptr(gr), T, n, H, _DTYPES[dtype]) != 0:
            raise ValueError(f"unsupported n={n} or dtype={dtype}")
        return gx, gy, gp, gr

    def post_sigmoid_fwd(self, x, y, mix, alpha, b, res, dtype: str = "bf16") -> np.ndarray:
        """post_fwd with post = sigmoid(alpha * mix + b); [T,n,H]."""
        mix, alpha, b = self._coeffs(mix, alpha, b)
        x, y, _, res, T, n, H = self._post_args(x, y, mix, res)
        out = np.empty((T, n, H), dtype=np.uint16)
        if self.lib.oracle_post_sigmoid_fwd(_ptr(x), _ptr(y), _ptr(mix), _ptr(alpha), _ptr(b), _ptr(res),
                                            _ptr(out), T, n, H, _DTYPES[dtype]) != 0:
            raise ValueError(f"unsupported n={n} or dtype={dtype}")
        return out

    def post_sigmoid_bwd(self, g, x, y, mix, alpha, b, res, dtype: str = "bf16"):
        """(grad_x [T,n,H], grad_y [T,H], grad_z float32 [T,n], grad_mix float32 [T,n],
        grad_res float32 [T,n,n])."""
        mix, alpha, b = self._coeffs(mix, alpha, b)
        x, y, _, res, T, n, H = self._post_args(x, y, mix, res)
        g = _as(g, np.uint16)
        if g.shape != (T, n, H):
            raise ValueError(f"g must be [{T},{n},{H}]")
        gx = np.empty((T, n, H), dtype=np.uint16)
        gy = np.empty((T, H), dtype=np.uint16)
        gz = np.empty((T, n), dtype=np.float32)
        gm = np.empty((T, n), dtype=np.float32)
        gr = np.empty((T, n, n), dtype=np.float32)
        if self.lib.oracle_post_sigmoid_bwd(_ptr(g), _ptr(x), _ptr(y), _ptr(mix), _ptr(alpha), _ptr(b),
                                            _ptr(res), _ptr(gx), _ptr(gy), _ptr(gz), _ptr(gm), _ptr(gr),
                                            T, n, H, _DTYPES[dtype]) != 0:
            raise ValueError(f"unsupported n={n} or dtype={dtype}")
        return gx, gy, gz, gm, gr

    def fwd(self, residual, pre) -> np.ndarray:
        """out[t,h] = bf16((pre0*r0 + pre1*r1) + (pre2*r2 + pre3*r3)); uint16 [T,H]."""
        residual = _as(residual, np.uint16)
        pre = _as(pre, np.float32)
        T, H = _shape_TH(residual)
        if pre.shape != (T, 4):
            raise ValueError(f"pre must be [{T},4], got {pre.shape}")
        out = np.empty((T, H), dtype=np.uint16)
        self.lib.oracle_h_aggregate_fwd(_ptr(residual), _ptr(pre), _ptr(out), T, H)
        return out

    def grad_residual(self, g, pre) -> np.ndarray:
        """grad_residual[t,k,h] = bf16(fp32(pre[t,k] * g[t,h])); uint16 [T,4,H]."""
        g = _as(g, np.uint16)
        pre = _as(pre, np.float32)
        T, H = g.shape
        if pre.shape != (T, 4):
            raise ValueError(f"pre must be [{T},4], got {pre.shape}")
        out = np.empty((T, 4, H), dtype=np.uint16)
        self.lib.oracle_h_aggregate_bwd_grad_residual(_ptr(g), _ptr(pre), _ptr(out), T, H)
        return out

    def grad_pre(self, g, residual) -> np.ndarray:
        """grad_pre[t,k] = sum_h g[t,h]*r[t,k,h] in FP32, ORDER-256; float32 [T,4]."""
        g = _as(g, np.uint16)
        residual = _as(residual, np.uint16)
        T, H = _shape_TH(residual)
        if g.shape != (T, H):
            raise ValueError(f"g must be [{T},{H}], got {g.shape}")
        out = np.empty((T, 4), dtype=np.float32)
        self.lib.oracle_h_aggregate_bwd_grad_pre(_ptr(g), _ptr(residual), _ptr(out), T, H)
        return out

    def bwd(self, g, residual, pre) -> tuple[np.ndarray, np.ndarray]:
        """(grad_residual uint16 [T,4,H], grad_pre float32 [T,4])."""
        g = _as(g, np.uint16)
        residual = _as(residual, np.uint16)
        pre = _as(pre, np.float32)
        T, H = _shape_TH(residual)
        if g.shape != (T, H) or pre.shape != (T, 4):
            raise ValueError("shape mismatch between g, residual and pre")
        gr = np.empty((T, 4, H), dtype=np.uint16)
        gp = np.empty((T, 4), dtype=np.float32)
        self.lib.oracle_h_aggregate_bwd(_ptr(g), _ptr(residual), _ptr(pre), _ptr(gr), _ptr(gp),
                                        T, H)
        return gr, gp


def default() -> Oracle:
    """The oracle built from ``mhc_oracle.c`` beside this file."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def bf16_from_float(x):
    return default().bf16_from_float(x)


def float_from_bf16(x):
    return default().float_from_bf16(x)


def fwd(residual, pre):
    return default().fwd(residual, pre)


def grad_residual(g, pre):
    return default().grad_residual(g, pre)


def grad_pre(g, residual):
    return default().grad_pre(g, residual)


def bwd(g, residual, pre):
    return default().bwd(g, residual, pre)


def f16_from_float(x):
    return default().f16_from_float(x)


def float_from_f16(x):
    return default().float_from_f16(x)


def aggregate_fwd(residual, pre, dtype="bf16"):
    return default().aggregate_fwd(residual, pre, dtype)


def aggregate_bwd(g, residual, pre, dtype="bf16"):
    return default().aggregate_bwd(g, residual, pre, dtype)


def pre_sigmoid(mix, alpha, b):
    return default().pre_sigmoid(mix, alpha, b)


def aggregate_sigmoid_fwd(residual, mix, alpha, b, dtype="bf16"):
    return default().aggregate_sigmoid_fwd(residual, mix, alpha, b, dtype)


def aggregate_sigmoid_bwd(g, residual, mix, alpha, b, dtype="bf16"):
    return default().aggregate_sigmoid_bwd(g, residual, mix, alpha, b, dtype)


def sigmoid_param_grad(grad_z, mix):
    return default().sigmoid_param_grad(grad_z, mix)


def post_fwd(x, y, post, res, dtype="bf16"):
    return default().post_fwd(x, y, post, res, dtype)


def post_bwd(g, x, y, post, res, dtype="bf16"):
    return default().post_bwd(g, x, y, post, res, dtype)


def post_sigmoid_fwd(x, y, mix, alpha, b, res, dtype="bf16"):
    return default().post_sigmoid_fwd(x, y, mix, alpha, b, res, dtype)


def post_sigmoid_bwd(g, x, y, mix, alpha, b, res, dtype="bf16"):
    return default().post_sigmoid_bwd(g, x, y, mix, alpha, b, res, dtype)

"""Device-buffer helpers for the GPU parity tests.

``DevBuf`` places data at a chosen byte offset from a 256-byte boundary inside
a larger allocation filled with a canary byte, so a test can force each kernel
path (16-, 4- or 2-byte alignment) and check afterwards that nothing outside
the buffer was written.  Calls go through the C ABI (``binding.*_raw``).
"""

from __future__ import annotations

import hashlib

import numpy as np
import torch

from invariant_mhc_aggregate_gb300 import _build, binding

GUARD = 512
CANARY = 0xA5


def lib():
    _build.build()
    return binding.load()


class DevBuf:
    def __init__(self, nbytes: int, offset: int = 0, device="cuda"):
        self.nbytes = int(nbytes)
        self.buf = torch.full((self.nbytes + 2 * GUARD + 256,), CANARY, dtype=torch.uint8,
                              device=device)
        base = self.buf.data_ptr()
        self.start = ((base + GUARD + 255) // 256) * 256 - base + offset
        self.ptr = base + self.start

    @classmethod
    def of(cls, t: torch.Tensor, offset: int = 0) -> "DevBuf":
        t = t.contiguous()
        b = cls(t.numel() * t.element_size(), offset)
        b.set(t)
        return b

    def view_bytes(self) -> torch.Tensor:
        return self.buf[self.start:self.start + self.nbytes]

    def set(self, t: torch.Tensor):
        src = t.contiguous().reshape(-1).view(torch.uint8)
        self.view_bytes().copy_(src.to(self.buf.device))

    def get(self, dtype=np.uint16, shape=None) -> np.ndarray:
        a = self.view_bytes().cpu().numpy().view(dtype)
        return a.reshape(shape) if shape is not None else a

    def guards_ok(self) -> bool:
        host = self.buf.cpu().numpy()
        return bool(np.all(host[:self.start] == CANARY)
                    and np.all(host[self.start + self.nbytes:] == CANARY))


def _align_of(offset: int) -> int:
    """Alignment of a DevBuf placed at `offset` bytes past a 256-byte boundary."""
    if offset == 0:
        return 256
    return offset & -offset


#: rows of at least this many values that neither a vector path nor the 4-byte
#: pair path takes use the realigned 16-byte path
SHIFT_MIN_H = 64


def expected_fwd_path(H: int, offsets) -> int:
    a = min(_align_of(offsets[0]), _align_of(offsets[2]))
    if H % 16 == 0 and a >= 32:
        return binding.MHC_PATH_VEC32
    if H % 8 == 0 and a >= 16:
        return binding.MHC_PATH_VEC16
    if H % 2 == 0 and a >= 4:
        return binding.MHC_PATH_PAIR
    if SHIFT_MIN_H <= H < 2 ** 30:
        return binding.MHC_PATH_SHIFT16
    return binding.MHC_PATH_ELEMENT


def expected_bwd_path(H: int, offsets) -> int:
    """The backward prefers the realigned path to the 4-byte pair path."""
    a = min(_align_of(offsets[0]), _align_of(offsets[1]), _align_of(offsets[3]))
    if H % 16 == 0 and a >= 32:
        return binding.MHC_PATH_VEC32
    if H % 8 == 0 and a >= 16:
        return binding.MHC_PATH_VEC16
    if SHIFT_MIN_H <= H < 2 ** 30:
        return binding.MHC_PATH_SHIFT16
    if H % 2 == 0 and a >= 4:
        return binding.MHC_PATH_PAIR
    return binding.MHC_PATH_ELEMENT


def stream_handle() -> int:
    return int(torch.cuda.current_stream().cuda_stream)


def run_fwd(residual: torch.Tensor, pre: torch.Tensor, offsets=(0, 0, 0), check_guards=True,
            expect_path="auto") -> np.ndarray:
    """Forward through the C ABI with residual / pre / out at the given byte offsets;
    checks that the library picks the path the alignment calls for."""
    T, _, H = residual.shape
    if expect_path == "auto":
        expect_path = expected_fwd_path(H, offsets)
    r = DevBuf.of(residual, offsets[0])
    p = DevBuf.of(pre, offsets[1])
    o = DevBuf(T * H * 2, offsets[2])
    if expect_path is not None:
        assert binding.fwd_path_raw(r.ptr, p.ptr, o.ptr, T, H) == expect_path
    st = binding.fwd_raw(r.ptr, p.ptr, o.ptr, T, H, stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    if check_guards:
        assert o.guards_ok(), "forward wrote outside out"
    return o.get(np.uint16, (T, H))


def run_bwd(g: torch.Tensor, residual: torch.Tensor, pre: torch.Tensor,
            offsets=(0, 0, 0, 0, 0), check_guards=True, expect_path="auto"):
    T, _, H = residual.shape
    if expect_path == "auto":
        expect_path = expected_bwd_path(H, offsets)
    gb = DevBuf.of(g, offsets[0])
    r = DevBuf.of(residual, offsets[1])
    p = DevBuf.of(pre, offsets[2])
    gr = DevBuf(T * 4 * H * 2, offsets[3])
    gp = DevBuf(T * 4 * 4, offsets[4])
    if expect_path is not None:
        assert binding.bwd_path_raw(gb.ptr, r.ptr, p.ptr, gr.ptr, gp.ptr, T, H) == expect_path
    st = binding.bwd_raw(gb.ptr, r.ptr, p.ptr, gr.ptr, gp.ptr, T, H, stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    if check_guards:
        assert gr.guards_ok() and gp.guards_ok(), "backward wrote outside its outputs"
    return gr.get(np.uint16, (T, 4, H)), gp.get(np.float32, (T, 4))


def u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def f32(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().numpy()


def sha(a) -> str:
    if isinstance(a, torch.Tensor):
        a = a.contiguous().cpu().view(torch.uint8).numpy()
    return hashlib.sha256(np.ascontiguousarray(a).tobytes()).hexdigest()


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str):
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    gv = got.view(np.uint8).reshape(got.shape + (-1,))
    wv = want.view(np.uint8).reshape(want.shape + (-1,))
    bad = np.nonzero(np.any(gv != wv, axis=-1))
    n = len(bad[0])
    if n:
        idx = tuple(int(b[0]) for b in bad)
        raise AssertionError(f"{what}: {n} elements differ, first at {idx}: "
                             f"got {got[idx]!r} want {want[idx]!r}")


DTYPE_CODE = {torch.bfloat16: binding.MHC_DTYPE_BF16, torch.float16: binding.MHC_DTYPE_F16}
DTYPE_NAME = {torch.bfloat16: "bf16", torch.float16: "f16"}


def run_agg_fwd(residual: torch.Tensor, pre: torch.Tensor, offsets=(0, 0, 0), check_guards=True):
    """General forward (stream count from residual.shape[1], storage from its dtype)
    through the C ABI with buffers at the given byte offsets."""
    T, n, H = residual.shape
    r = DevBuf.of(residual, offsets[0])
    p = DevBuf.of(pre, offsets[1])
    o = DevBuf(T * H * 2, offsets[2])
    assert binding.agg_fwd_path_raw(r.ptr, p.ptr, o.ptr, T, n, H) == expected_fwd_path(H, offsets)
    st = binding.agg_fwd_raw(r.ptr, p.ptr, o.ptr, T, n, H, DTYPE_CODE[residual.dtype], stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    if check_guards:
        assert o.guards_ok(), "forward wrote outside out"
    return o.get(np.uint16, (T, H))


def run_agg_bwd(g: torch.Tensor, residual: torch.Tensor, pre: torch.Tensor,
                offsets=(0, 0, 0, 0, 0), check_guards=True):
    T, n, H = residual.shape
    gb = DevBuf.of(g, offsets[0])
    r = DevBuf.of(residual, offsets[1])
    p = DevBuf.of(pre, offsets[2])
    gr = DevBuf(T * n * H * 2, offsets[3])
    gp = DevBuf(T * n * 4, offsets[4])
    assert binding.agg_bwd_path_raw(gb.ptr, r.ptr, p.ptr, gr.ptr, gp.ptr, T, n, H) == \
        expected_bwd_path(H, offsets)
    st = binding.agg_bwd_raw(gb.ptr, r.ptr, p.ptr, gr.ptr, gp.ptr, T, n, H,
                             DTYPE_CODE[residual.dtype], stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    if check_guards:
        assert gr.guards_ok() and gp.guards_ok(), "backward wrote outside its outputs"
    return gr.get(np.uint16, (T, n, H)), gp.get(np.float32, (T, n))

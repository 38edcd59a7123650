"""The bounded waits of the bulk-copy kernels: a wait on a shared-memory
barrier that nothing completes gives up after its time limit (about 1 s) and
reports it, so that the GPU never hangs, and the CUDA context stays usable;
the library's own counter of such timeouts stays at zero in normal runs."""

import ctypes
import os
import subprocess

import pytest
import torch

from _gpu import lib
from invariant_mhc_aggregate_gb300 import _build, binding
from invariant_mhc_aggregate_gb300.inputs import backward_inputs, post_inputs

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe(tmp_path_factory):
    lib()
    so = str(tmp_path_factory.mktemp("wait_probe") / "wait_probe.so")
    cmd = [_build.nvcc_path(), *_build.NVCC_FLAGS, "-shared", "-I", _build.CSRC, "-o", so,
           os.path.join(HERE, "wait_probe.cu")]
    subprocess.run(cmd, check=True, capture_output=True)
    p = ctypes.CDLL(so)
    p.run_wait_probe.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    p.run_wait_probe.restype = ctypes.c_int
    return p


def _run(probe, arrive: int):
    result = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    elapsed = torch.zeros((1,), dtype=torch.int64, device="cuda")
    assert probe.run_wait_probe(arrive, result.data_ptr(), elapsed.data_ptr()) == 0
    return int(result.item()), int(elapsed.item())


def test_completed_barrier_wait_returns_at_once(probe):
    done, ns = _run(probe, 1)
    assert done == 1
    assert ns < 10_000_000


def test_wait_that_never_completes_gives_up(probe):
    done, ns = _run(probe, 0)
    assert done == 0
    assert 1_000_000_000 <= ns < 5_000_000_000, ns
    # the context is still usable: a library call after it gives correct results
    x, y, post, res, g = (t.cuda() for t in post_inputs(8, 4096, 4, "normal", 11, with_grad=True))
    gx, gy, gp, gr = binding.post_backward(g, x, y, post, res)
    gx2, gy2, gp2, gr2 = binding.post_backward(g, x, y, post, res)
    assert torch.equal(gx.view(torch.int16), gx2.view(torch.int16))
    assert binding.wait_timeouts() == 0


def test_library_counts_no_timeouts_in_normal_runs():
    assert binding.wait_timeouts() >= 0    # reset
    for n in (1, 2, 4):
        x, y, post, res, g = (t.cuda() for t in post_inputs(300, 7168, n, "normal", 12 + n, with_grad=True))
        binding.post_backward(g, x, y, post, res)
    # the aggregate backward's bulk-copy kernel (odd H)
    g, res, pre = (t.cuda() for t in backward_inputs(300, 7167, "normal", 16))
    binding.aggregate_backward(g, res, pre)
    assert binding.wait_timeouts() == 0

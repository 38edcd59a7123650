"""The library used from plain C: tests/c_consumer.c is compiled with gcc
against the CUDA runtime and libmhc_h_aggregate.so (no Python or PyTorch in
the process), runs the forward and the backward through the C ABI, and its
outputs must equal the oracle's bytes."""

import os
import subprocess

import numpy as np
import pytest

import oracle
from invariant_mhc_aggregate_gb300 import _build
from invariant_mhc_aggregate_gb300.inputs import backward_inputs, as_u16, as_f32

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.mark.parametrize("T,H", [(37, 7168), (5, 1279)])
def test_c_program_through_the_abi(tmp_path, T, H):
    _build.build()
    exe = tmp_path / "c_consumer"
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-o", str(exe),
                    os.path.join(HERE, "c_consumer.c"), "-I", _build.INCLUDE, "-I", f"{CUDA}/include",
                    "-L", _build.LIB_DIR, "-lmhc_h_aggregate", "-L", f"{CUDA}/lib64", "-lcudart",
                    f"-Wl,-rpath,{_build.LIB_DIR}", f"-Wl,-rpath,{CUDA}/lib64"], check=True)
    g, res, pre = backward_inputs(T, H, "ragged", 300)
    g16, r16, pf = as_u16(g), as_u16(res), as_f32(pre)
    (tmp_path / "residual.bin").write_bytes(r16.tobytes())
    (tmp_path / "pre.bin").write_bytes(pf.tobytes())
    (tmp_path / "g.bin").write_bytes(g16.tobytes())
    res_run = subprocess.run([str(exe), str(tmp_path), str(T), str(H)], capture_output=True, text=True)
    assert res_run.returncode == 0, res_run.stderr
    out = np.frombuffer((tmp_path / "out.bin").read_bytes(), dtype=np.uint16).reshape(T, H)
    gr = np.frombuffer((tmp_path / "grad_residual.bin").read_bytes(), dtype=np.uint16).reshape(T, 4, H)
    gp = np.frombuffer((tmp_path / "grad_pre.bin").read_bytes(), dtype=np.float32).reshape(T, 4)
    assert np.array_equal(out, oracle.fwd(r16, pf))
    want_gr, want_gp = oracle.bwd(g16, r16, pf)
    assert np.array_equal(gr, want_gr)
    assert np.array_equal(gp.view(np.uint32), want_gp.view(np.uint32))

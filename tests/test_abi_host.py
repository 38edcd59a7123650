"""The C-ABI library on the host: it builds, loads, exports what the header
declares, picks paths and rejects bad arguments without touching a GPU."""

import ctypes
import os
import re
import subprocess

import pytest

from invariant_mhc_aggregate_gb300 import _build, binding

HEADER = os.path.join(_build.INCLUDE, "mhc_h_aggregate.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.load()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:MHC_API\s+)?(?:const\s+)?\w+\*?\s+\*?(mhc_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_binding_exports():
    assert tuple(header_functions()) == binding.EXPORTS


def test_every_declared_symbol_is_exported(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_exported_symbols_are_c_linkage():
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    names = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in header_functions():
        assert name in names, f"{name} not exported with C linkage"


def test_only_the_c_abi_is_exported():
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    names = {line.split()[-1] for line in out.splitlines() if line.strip()}
    assert names == set(header_functions()), sorted(names - set(header_functions()))[:10]


def test_abi_version(lib):
    assert lib.mhc_h_aggregate_abi_version() == 6


def test_status_strings(lib):
    for s in range(4):
        assert lib.mhc_status_string(s).decode().startswith("MHC_")
    assert b"unknown" in lib.mhc_status_string(99)


# --- path selection: pure host logic on addresses that are never dereferenced

A = 1 << 40          # a 256-byte aligned fake device address
GAP = 1 << 34        # keeps fake buffers apart


def fpath(r_off=0, p_off=0, o_off=0, T=4, H=4096):
    return binding.fwd_path_raw(A + r_off, A + GAP + p_off, A + 2 * GAP + o_off, T, H)


def bpath(g_off=0, r_off=0, p_off=0, gr_off=0, gp_off=0, T=4, H=4096):
    return binding.bwd_path_raw(A + g_off, A + GAP + r_off, A + 2 * GAP + p_off,
                                A + 3 * GAP + gr_off, A + 4 * GAP + gp_off, T, H)


def test_fwd_path_choice(lib):
    assert fpath() == binding.MHC_PATH_VEC32
    assert fpath(p_off=4) == binding.MHC_PATH_VEC32          # pre only needs 4 bytes
    assert fpath(r_off=16) == binding.MHC_PATH_VEC16
    assert fpath(o_off=16) == binding.MHC_PATH_VEC16
    assert fpath(H=4104) == binding.MHC_PATH_VEC16           # H % 16 == 8
    assert fpath(r_off=4) == binding.MHC_PATH_PAIR
    assert fpath(o_off=8) == binding.MHC_PATH_PAIR
    assert fpath(r_off=2) == binding.MHC_PATH_SHIFT16         # 2-byte aligned, H >= 64: realigned
    assert fpath(H=2050) == binding.MHC_PATH_PAIR
    assert fpath(H=1279) == binding.MHC_PATH_SHIFT16          # odd H >= 64: realigned
    assert fpath(H=4097) == binding.MHC_PATH_SHIFT16
    assert fpath(H=64, r_off=2) == binding.MHC_PATH_SHIFT16
    assert fpath(H=62) == binding.MHC_PATH_PAIR
    assert fpath(H=56, r_off=2) == binding.MHC_PATH_ELEMENT   # shorter rows: 2-byte path
    assert fpath(H=63) == binding.MHC_PATH_ELEMENT
    # the realigned path keeps row positions in 32 bits (H < 2^30); one token
    # so that the fake buffers stay apart
    assert fpath(H=(1 << 30) - 1, T=1) == binding.MHC_PATH_SHIFT16
    assert fpath(H=(1 << 30) + 1, T=1) == binding.MHC_PATH_ELEMENT
    assert fpath(r_off=1) == binding.MHC_PATH_NONE           # not BF16 aligned
    assert fpath(p_off=2) == binding.MHC_PATH_NONE           # not FP32 aligned
    assert fpath(T=0) == binding.MHC_PATH_NONE
    assert fpath(T=-1) == binding.MHC_PATH_NONE
    assert fpath(H=0) == binding.MHC_PATH_NONE


def test_bwd_path_choice(lib):
    assert bpath() == binding.MHC_PATH_VEC32
    assert bpath(p_off=4, gp_off=4) == binding.MHC_PATH_VEC32
    assert bpath(g_off=16) == binding.MHC_PATH_VEC16
    assert bpath(gr_off=16) == binding.MHC_PATH_VEC16
    assert bpath(H=4104) == binding.MHC_PATH_VEC16
    assert bpath(g_off=2) == binding.MHC_PATH_SHIFT16
    assert bpath(gr_off=4) == binding.MHC_PATH_SHIFT16          # the backward prefers the realigned path
    assert bpath(H=2050) == binding.MHC_PATH_SHIFT16
    assert bpath(H=2050, r_off=2) == binding.MHC_PATH_SHIFT16
    assert bpath(H=1279) == binding.MHC_PATH_SHIFT16
    assert bpath(H=50) == binding.MHC_PATH_PAIR
    assert bpath(H=50, r_off=2) == binding.MHC_PATH_ELEMENT
    assert bpath(H=13) == binding.MHC_PATH_ELEMENT
    assert bpath(gp_off=2) == binding.MHC_PATH_NONE
    assert bpath(T=0) == binding.MHC_PATH_NONE


def test_fwd_rejects_overlap(lib):
    T, H = 4, 64
    # out starts inside residual
    assert binding.fwd_path_raw(A, A + GAP, A + 16, T, H) == binding.MHC_PATH_NONE
    # out overlaps pre
    assert binding.fwd_path_raw(A, A + GAP, A + GAP + 32, T, H) == binding.MHC_PATH_NONE
    # out right after residual is fine
    assert binding.fwd_path_raw(A, A + GAP, A + T * 4 * H * 2, T, H) == binding.MHC_PATH_VEC32


def test_bwd_rejects_overlap(lib):
    T, H = 4, 64
    g, r, p = A, A + GAP, A + 2 * GAP
    assert binding.bwd_path_raw(g, r, p, r, A + 3 * GAP, T, H) == binding.MHC_PATH_NONE
    assert binding.bwd_path_raw(g, r, p, A + 3 * GAP, A + 3 * GAP + 64, T, H) == binding.MHC_PATH_NONE
    assert binding.bwd_path_raw(g, r, p, A + 3 * GAP, g, T, H) == binding.MHC_PATH_NONE


# --- entry points: rejected calls return before any CUDA call

def test_fwd_invalid_arguments(lib):
    ok = dict(residual=A, pre=A + GAP, out=A + 2 * GAP)
    assert binding.fwd_raw(ok["residual"], ok["pre"], ok["out"], -1, 8) == binding.MHC_ERR_INVALID_ARG
    assert binding.fwd_raw(ok["residual"], ok["pre"], ok["out"], 1, 0) == binding.MHC_ERR_INVALID_ARG
    assert binding.fwd_raw(0, ok["pre"], ok["out"], 1, 8) == binding.MHC_ERR_INVALID_ARG
    assert binding.fwd_raw(ok["residual"], 0, ok["out"], 1, 8) == binding.MHC_ERR_INVALID_ARG
    assert binding.fwd_raw(ok["residual"], ok["pre"], 0, 1, 8) == binding.MHC_ERR_INVALID_ARG
    assert binding.fwd_raw(ok["residual"] + 1, ok["pre"], ok["out"], 1, 8) == binding.MHC_ERR_INVALID_ARG
    assert binding.fwd_raw(ok["residual"], ok["pre"], ok["residual"], 1, 8) == binding.MHC_ERR_INVALID_ARG
    # byte count of residual overflows int64
    assert binding.fwd_raw(ok["residual"], ok["pre"], ok["out"], 1 << 32, 1 << 29) == binding.MHC_ERR_INVALID_ARG


def test_bwd_invalid_arguments(lib):
    args = [A, A + GAP, A + 2 * GAP, A + 3 * GAP, A + 4 * GAP]
    assert binding.bwd_raw(*args, -5, 8) == binding.MHC_ERR_INVALID_ARG
    assert binding.bwd_raw(*args, 1, -8) == binding.MHC_ERR_INVALID_ARG
    for i in range(5):
        bad = list(args)
        bad[i] = 0
        assert binding.bwd_raw(*bad, 2, 8) == binding.MHC_ERR_INVALID_ARG, i
    bad = list(args)
    bad[4] += 2
    assert binding.bwd_raw(*bad, 2, 8) == binding.MHC_ERR_INVALID_ARG


def test_zero_tokens_is_a_noop(lib):
    # T == 0 succeeds without a launch, even with NULL pointers
    assert binding.fwd_raw(0, 0, 0, 0, 4096) == binding.MHC_OK
    assert binding.bwd_raw(0, 0, 0, 0, 0, 0, 4096) == binding.MHC_OK
    assert lib.mhc_h_aggregate_last_cuda_error() == 0


# --- build settings

def test_build_has_no_fast_math():
    flags = " ".join(_build.NVCC_FLAGS)
    assert "use_fast_math" not in flags
    assert "--fmad=false" in flags and "-ftz=false" in flags
    assert "arch=compute_103a,code=sm_103a" in flags


def test_kernels_use_rn_intrinsics_only():
    src = "".join(open(p).read() for p in _build.DEPS if p.startswith(_build.CSRC))
    code = re.sub(r"//.*", "", src)
    assert "__fmaf" not in code and "fmaf(" not in code and "__fma_rn" not in code
    assert "fma.rn" not in code
    # one writer per output element: no device atomics or reductions on any
    # output; the only atomic is the bulk-copy ring's shared-memory counter of
    # warps that released a stage
    assert not re.findall(r"\batomic[A-Z]\w*\(", code)
    assert not re.search(r"\bred\.", code)
    atoms = re.findall(r"\batom\.[\w.:]+", code)
    assert atoms == ["atom.acq_rel.cta.shared::cta.inc.u32"]
    assert code.count("release_count(") == 2   # its definition and the stage ring's one call


def test_fastdiv_exhaustive_sample(tmp_path):
    """The launch-time divider in csrc/fastdiv.cuh, compiled as host C++."""
    prog = tmp_path / "fd.cpp"
    prog.write_text(r'''
#include "fastdiv.cuh"
#include <cstdio>
#include <cstdint>
int main() {
    uint64_t bad = 0, n_checked = 0;
    const uint32_t ds[] = {1u, 2u, 3u, 7u, 8u, 160u, 255u, 256u, 257u, 512u, 513u, 896u,
                           1279u, 2050u, 4097u, 7168u, 65535u, 65536u, 1000003u,
                           0x7FFFFFFFu, 0x80000000u, 0x80000001u, 0xFFFFFFFEu, 0xFFFFFFFFu};
    for (uint32_t d : ds) {
        FastDivU32 f = make_fastdiv_u32(d);
        uint64_t x = 0x9E3779B97F4A7C15ull;
        for (int i = 0; i < 200000; ++i) {
            x ^= x << 13; x ^= x >> 7; x ^= x << 17;
            uint32_t n = uint32_t(x);
            if (i < 4096) n = uint32_t(i);
            if (i >= 4096 && i < 8192) n = 0xFFFFFFFFu - uint32_t(i - 4096);
            if (i >= 8192 && i < 12288) n = uint32_t(uint64_t(d) * uint32_t(i - 8192) + (i & 1 ? d - 1 : 0));
            ++n_checked;
            if (fastdiv_u32(n, f) != n / d) { if (bad < 5) printf("d=%u n=%u\n", d, n); ++bad; }
        }
    }
    printf("checked %llu bad %llu\n", (unsigned long long)n_checked, (unsigned long long)bad);
    return bad != 0;
}
''')
    exe = tmp_path / "fd"
    subprocess.run(["g++", "-std=c++17", "-O2", "-I", _build.CSRC, "-o", str(exe), str(prog)],
                   check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout


# --- the general entry points (stream count n, storage dtype)

def test_general_path_choice(lib):
    def gpath(n, H=4096, r_off=0, o_off=0, T=4):
        return binding.agg_fwd_path_raw(A + r_off, A + GAP, A + 2 * GAP + o_off, T, n, H)
    for n in (1, 2, 4, 8):
        assert gpath(n) == binding.MHC_PATH_VEC32
        assert gpath(n, r_off=16) == binding.MHC_PATH_VEC16
        assert gpath(n, H=2050) == binding.MHC_PATH_PAIR
        assert gpath(n, H=1279) == binding.MHC_PATH_SHIFT16
        assert gpath(n, H=34) == binding.MHC_PATH_PAIR
        assert gpath(n, H=33) == binding.MHC_PATH_ELEMENT
    for n in (0, 3, 5, 16, -1):
        assert gpath(n) == binding.MHC_PATH_NONE
    # n = 4 is the pages' op
    assert gpath(4) == binding.fwd_path_raw(A, A + GAP, A + 2 * GAP, 4, 4096)
    # an output that ends where an n = 8 residual would still be: overlap depends on n
    T, H = 2, 64
    out_at = A + T * 4 * H * 2
    assert binding.agg_fwd_path_raw(A, A + GAP, out_at, T, 4, H) != binding.MHC_PATH_NONE
    assert binding.agg_fwd_path_raw(A, A + GAP, out_at, T, 8, H) == binding.MHC_PATH_NONE


def test_general_bwd_path_choice(lib):
    for n in (1, 2, 4, 8):
        assert binding.agg_bwd_path_raw(A, A + GAP, A + 2 * GAP, A + 3 * GAP, A + 4 * GAP, 4, n,
                                        4096) == binding.MHC_PATH_VEC32
    assert binding.agg_bwd_path_raw(A, A + GAP, A + 2 * GAP, A + 3 * GAP, A + 4 * GAP, 4, 6,
                                    4096) == binding.MHC_PATH_NONE


def test_general_invalid_arguments(lib):
    args = (A, A + GAP, A + 2 * GAP)
    assert binding.agg_fwd_raw(*args, 4, 3, 64, binding.MHC_DTYPE_BF16) == binding.MHC_ERR_UNSUPPORTED
    assert binding.agg_fwd_raw(*args, 4, 4, 64, 7) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_fwd_raw(*args, -1, 2, 64, binding.MHC_DTYPE_F16) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_fwd_raw(*args, 0, 8, 64, binding.MHC_DTYPE_F16) == binding.MHC_OK
    bargs = (A, A + GAP, A + 2 * GAP, A + 3 * GAP, A + 4 * GAP)
    assert binding.agg_bwd_raw(*bargs, 4, 0, 64, binding.MHC_DTYPE_BF16) == binding.MHC_ERR_UNSUPPORTED
    assert binding.agg_bwd_raw(*bargs, 4, 2, 64, 2) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_bwd_raw(*bargs, 0, 1, 64, binding.MHC_DTYPE_BF16) == binding.MHC_OK
    # byte count of an n = 8 residual overflows int64
    assert binding.agg_fwd_raw(*args, 1 << 31, 8, 1 << 29, binding.MHC_DTYPE_BF16) == binding.MHC_ERR_INVALID_ARG


# --- the pre coefficients computed from the mix (sigmoid): rejected calls

def test_pre_sigmoid_invalid_arguments(lib):
    mix, alpha, b, pre = A, A + GAP, A + 2 * GAP, A + 3 * GAP
    assert binding.pre_sigmoid_raw(mix, alpha, b, pre, 4, 3) == binding.MHC_ERR_UNSUPPORTED
    assert binding.pre_sigmoid_raw(mix, alpha, b, pre, -1, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.pre_sigmoid_raw(0, 0, 0, 0, 0, 4) == binding.MHC_OK
    assert binding.pre_sigmoid_raw(0, alpha, b, pre, 4, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.pre_sigmoid_raw(mix, 0, b, pre, 4, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.pre_sigmoid_raw(mix, alpha, 0, pre, 4, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.pre_sigmoid_raw(mix, alpha, b + 2, pre, 4, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.pre_sigmoid_raw(mix, alpha, b, mix + 16, 4, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.pre_sigmoid_raw(mix, alpha, pre + 8, pre, 4, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.pre_sigmoid_raw(mix, pre + 60, b, pre, 4, 4) == binding.MHC_ERR_INVALID_ARG


def test_aggregate_sigmoid_fwd_invalid_arguments(lib):
    r, mix, alpha, b, out = A, A + GAP, A + 2 * GAP, A + 3 * GAP, A + 4 * GAP
    bf16 = binding.MHC_DTYPE_BF16
    assert binding.agg_sigmoid_fwd_raw(r, mix, alpha, b, out, 4, 4, 64, 7) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_sigmoid_fwd_raw(r, mix, alpha, b, out, 4, 3, 64, bf16) == binding.MHC_ERR_UNSUPPORTED
    assert binding.agg_sigmoid_fwd_raw(0, 0, 0, 0, 0, 0, 4, 64, bf16) == binding.MHC_OK
    assert binding.agg_sigmoid_fwd_raw(r, mix, 0, b, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_sigmoid_fwd_raw(r, mix, alpha, 0, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_sigmoid_fwd_raw(r, mix, alpha, b + 1, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_sigmoid_fwd_raw(r, mix, out + 64, b, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_sigmoid_fwd_raw(r, mix, alpha, out + 4, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.agg_sigmoid_fwd_raw(r, out, alpha, b, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG


def test_aggregate_sigmoid_bwd_invalid_arguments(lib):
    g, r, mix, alpha, b = A, A + GAP, A + 2 * GAP, A + 3 * GAP, A + 4 * GAP
    gr, gz, gm = A + 5 * GAP, A + 6 * GAP, A + 7 * GAP
    bf16 = binding.MHC_DTYPE_BF16

    def call(**kw):
        a = dict(g=g, r=r, mix=mix, alpha=alpha, b=b, gr=gr, gz=gz, gm=gm, T=4, n=4, H=64, dt=bf16)
        a.update(kw)
        return binding.agg_sigmoid_bwd_raw(a["g"], a["r"], a["mix"], a["alpha"], a["b"], a["gr"],
                                           a["gz"], a["gm"], a["T"], a["n"], a["H"], a["dt"])

    assert call(n=6) == binding.MHC_ERR_UNSUPPORTED
    assert call(dt=5) == binding.MHC_ERR_INVALID_ARG
    assert call(T=0, g=0, r=0, mix=0, alpha=0, b=0, gr=0, gz=0, gm=0) == binding.MHC_OK
    for name in ("g", "r", "mix", "alpha", "b", "gr", "gz", "gm"):
        assert call(**{name: 0}) == binding.MHC_ERR_INVALID_ARG, name
    assert call(gm=gm + 2) == binding.MHC_ERR_INVALID_ARG
    assert call(gm=gz + 32) == binding.MHC_ERR_INVALID_ARG        # grad_mix overlaps grad_z
    assert call(gm=mix) == binding.MHC_ERR_INVALID_ARG            # grad_mix overlaps mix
    assert call(gm=gr + 128) == binding.MHC_ERR_INVALID_ARG       # grad_mix overlaps grad_residual
    assert call(gz=mix + 16) == binding.MHC_ERR_INVALID_ARG       # grad_z overlaps mix
    assert call(b=gz + 8) == binding.MHC_ERR_INVALID_ARG          # b overlaps grad_z
    assert call(alpha=gm) == binding.MHC_ERR_INVALID_ARG          # alpha overlaps grad_mix
    assert call(alpha=gr + 2 * 64) == binding.MHC_ERR_INVALID_ARG  # alpha inside grad_residual


def test_sigmoid_param_grad_invalid_arguments(lib):
    gz, mix, gb, ga = A, A + GAP, A + 2 * GAP, A + 3 * GAP
    assert binding.sigmoid_param_grad_raw(gz, mix, gb, ga, 8, 5) == binding.MHC_ERR_UNSUPPORTED
    assert binding.sigmoid_param_grad_raw(gz, mix, gb, ga, -1, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.sigmoid_param_grad_raw(gz, mix, 0, ga, 8, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.sigmoid_param_grad_raw(gz, mix, gb, 0, 8, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.sigmoid_param_grad_raw(0, mix, gb, ga, 8, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.sigmoid_param_grad_raw(gz, 0, gb, ga, 8, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.sigmoid_param_grad_raw(gz, mix, gb, gb + 12, 8, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.sigmoid_param_grad_raw(gz, mix, gz + 64, ga, 8, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.sigmoid_param_grad_raw(gz, mix, gb, mix + 4, 8, 4) == binding.MHC_ERR_INVALID_ARG
    assert binding.sigmoid_param_grad_raw(gz, mix, gb + 2, ga, 8, 4) == binding.MHC_ERR_INVALID_ARG


# --- mHC post: path choice and rejected calls

def post_fpath(x_off=0, y_off=0, p_off=0, r_off=0, o_off=0, T=4, n=4, H=4096):
    return binding.post_fwd_path_raw(A + x_off, A + GAP + y_off, A + 2 * GAP + p_off,
                                     A + 3 * GAP + r_off, A + 4 * GAP + o_off, T, n, H)


def post_bpath(offs=(0,) * 9, T=4, n=4, H=4096):
    return binding.post_bwd_path_raw(*(A + i * GAP + o for i, o in enumerate(offs)), T, n, H)


def test_post_fwd_path_choice(lib):
    assert post_fpath() == binding.MHC_PATH_VEC16
    assert post_fpath(p_off=4, r_off=4) == binding.MHC_PATH_VEC16     # coefficients need 4 bytes
    assert post_fpath(y_off=16) == binding.MHC_PATH_VEC16
    assert post_fpath(o_off=16) == binding.MHC_PATH_VEC16
    assert post_fpath(H=4104) == binding.MHC_PATH_VEC16
    assert post_fpath(x_off=8) == binding.MHC_PATH_ELEMENT
    assert post_fpath(o_off=8) == binding.MHC_PATH_ELEMENT
    assert post_fpath(H=4100) == binding.MHC_PATH_ELEMENT
    assert post_fpath(H=1279, n=8) == binding.MHC_PATH_ELEMENT
    assert post_fpath(x_off=1) == binding.MHC_PATH_NONE
    assert post_fpath(r_off=2) == binding.MHC_PATH_NONE
    assert post_fpath(n=3) == binding.MHC_PATH_NONE
    assert post_fpath(T=0) == binding.MHC_PATH_NONE


def test_post_bwd_path_choice(lib):
    assert post_bpath() == binding.MHC_PATH_VEC16
    assert post_bpath(H=4104) == binding.MHC_PATH_VEC16
    for i in range(5):   # any 2-byte buffer off 16 bytes: the 2-byte path
        offs = [0] * 9
        offs[i if i < 3 else i + 2] = 8
        assert post_bpath(tuple(offs)) == binding.MHC_PATH_ELEMENT, i
    assert post_bpath(H=4100) == binding.MHC_PATH_ELEMENT
    assert post_bpath((0, 0, 0, 0, 0, 0, 0, 2, 0)) == binding.MHC_PATH_NONE
    assert post_bpath(T=0) == binding.MHC_PATH_NONE


def test_post_rejects_overlap(lib):
    T, n, H = 4, 4, 64
    x, y, p, r, o = A, A + GAP, A + 2 * GAP, A + 3 * GAP, A + 4 * GAP
    assert binding.post_fwd_path_raw(x, y, p, r, x + 64, T, n, H) == binding.MHC_PATH_NONE
    assert binding.post_fwd_path_raw(x, y, p, r, y, T, n, H) == binding.MHC_PATH_NONE
    assert binding.post_fwd_path_raw(x, y, p, o + 256, o, T, n, H) == binding.MHC_PATH_NONE
    assert binding.post_fwd_path_raw(x, y, p, r, x + T * n * H * 2, T, n, H) == binding.MHC_PATH_VEC16
    bufs = [A + i * GAP for i in range(9)]
    # every output against every other buffer
    for out in range(5, 9):
        for other in range(9):
            if other == out:
                continue
            b = list(bufs)
            b[out] = b[other] + 16
            assert binding.post_bwd_path_raw(*b, T, n, H) == binding.MHC_PATH_NONE, (out, other)


def test_post_invalid_arguments(lib):
    bf16 = binding.MHC_DTYPE_BF16
    f = [A + i * GAP for i in range(5)]
    assert binding.post_fwd_raw(*f, 4, 3, 64, bf16) == binding.MHC_ERR_UNSUPPORTED
    assert binding.post_fwd_raw(*f, 4, 4, 64, 9) == binding.MHC_ERR_INVALID_ARG
    assert binding.post_fwd_raw(*f, -1, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.post_fwd_raw(*f, 4, 4, 0, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.post_fwd_raw(0, 0, 0, 0, 0, 0, 4, 64, bf16) == binding.MHC_OK
    for i in range(5):
        bad = list(f)
        bad[i] = 0
        assert binding.post_fwd_raw(*bad, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG, i
    b = [A + i * GAP for i in range(9)]
    assert binding.post_bwd_raw(*b, 4, 5, 64, bf16) == binding.MHC_ERR_UNSUPPORTED
    assert binding.post_bwd_raw(*b, 4, 4, 64, -1) == binding.MHC_ERR_INVALID_ARG
    assert binding.post_bwd_raw(*([0] * 9), 0, 2, 64, binding.MHC_DTYPE_F16) == binding.MHC_OK
    for i in range(9):
        bad = list(b)
        bad[i] = 0
        assert binding.post_bwd_raw(*bad, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG, i
    bad = list(b)
    bad[8] += 2      # grad_res not FP32 aligned
    assert binding.post_bwd_raw(*bad, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    # byte count of an n = 8 x overflows int64
    assert binding.post_fwd_raw(*f, 1 << 31, 8, 1 << 29, bf16) == binding.MHC_ERR_INVALID_ARG
    assert lib.mhc_h_aggregate_last_cuda_error() == 0


def test_post_sigmoid_invalid_arguments(lib):
    bf16 = binding.MHC_DTYPE_BF16
    x, y, mix, alpha, b, res, out = (A + i * GAP for i in range(7))
    assert binding.post_sigmoid_fwd_raw(x, y, mix, alpha, b, res, out, 4, 3, 64, bf16) == binding.MHC_ERR_UNSUPPORTED
    assert binding.post_sigmoid_fwd_raw(x, y, mix, alpha, b, res, out, 4, 4, 64, 5) == binding.MHC_ERR_INVALID_ARG
    assert binding.post_sigmoid_fwd_raw(0, 0, 0, 0, 0, 0, 0, 0, 4, 64, bf16) == binding.MHC_OK
    assert binding.post_sigmoid_fwd_raw(x, y, mix, 0, b, res, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.post_sigmoid_fwd_raw(x, y, mix, alpha, b + 2, res, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.post_sigmoid_fwd_raw(x, y, mix, out + 64, b, res, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    assert binding.post_sigmoid_fwd_raw(x, y, out + 16, alpha, b, res, out, 4, 4, 64, bf16) == binding.MHC_ERR_INVALID_ARG
    names = ("g", "x", "y", "mix", "alpha", "b", "res", "gx", "gy", "gz", "gm", "gr")
    base = {nm: A + i * GAP for i, nm in enumerate(names)}

    def call(**kw):
        a = dict(base, T=4, n=4, H=64, dt=bf16)
        a.update(kw)
        return binding.post_sigmoid_bwd_raw(*(a[nm] for nm in names), a["T"], a["n"], a["H"], a["dt"])

    assert call(n=6) == binding.MHC_ERR_UNSUPPORTED
    assert call(dt=3) == binding.MHC_ERR_INVALID_ARG
    for nm in names:
        assert call(**{nm: 0}) == binding.MHC_ERR_INVALID_ARG, nm
    assert call(gm=base["gm"] + 2) == binding.MHC_ERR_INVALID_ARG
    for out in ("gx", "gy", "gz", "gm", "gr"):
        for other in names:
            if other != out:
                assert call(**{out: base[other]}) == binding.MHC_ERR_INVALID_ARG, (out, other)
    assert call(alpha=base["gz"] + 4) == binding.MHC_ERR_INVALID_ARG
    assert call(b=base["gm"]) == binding.MHC_ERR_INVALID_ARG


def test_post_vector_index_limit(lib):
    """Rows of 2^31 16-byte vectors or more are rejected on the vector path
    (the kernels index vectors of a row in 32 bits); buffers spaced 2^36 apart
    so that they stay disjoint."""
    big = 1 << 36
    bf16 = binding.MHC_DTYPE_BF16
    H = 1 << 34                       # H / 8 = 2^31 vectors
    f = [A + i * big for i in range(5)]
    assert binding.post_fwd_path_raw(*f, 1, 1, H) == binding.MHC_PATH_VEC16
    assert binding.post_fwd_raw(*f, 1, 1, H, bf16) == binding.MHC_ERR_UNSUPPORTED
    b = [A + i * big for i in range(9)]
    assert binding.post_bwd_raw(*b, 1, 1, H, bf16) == binding.MHC_ERR_UNSUPPORTED

"""The realigned 16-byte path (rows of H >= 64 that no vector path takes):
every row phase, segment edges and buffer ends, against the oracle byte for
byte, with guard bands around every output.

Rows that start part-way into a 16-byte line are read and written with
aligned 16-byte accesses and realigned in registers; the path must give the
same bytes as every other path ("Add batch-invariant h_aggregate kernel",
Batch invariance) and write nothing outside its rows.
"""

import numpy as np
import pytest
import torch

import oracle
from _gpu import DTYPE_NAME, assert_bytes_equal, lib, run_agg_bwd, run_agg_fwd, u16, f32
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.inputs import backward_inputs

pytestmark = pytest.mark.gpu

# 64 is the smallest H on the path; 2048 / 4096 are the backward / forward
# segment lengths (2048 for the n = 8 forward)
HS = (64, 65, 127, 2047, 2048, 2049, 4095, 4097, 6143, 8193)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


@pytest.mark.parametrize("H", HS)
def test_every_phase_forward(H):
    T, n = 3, 4
    _, res, pre = backward_inputs(T, H, "ragged", 300 + H, n=n)
    want = oracle.aggregate_fwd(u16(res), f32(pre), "bf16")
    for r_off in range(0, 16, 2):
        o_off = (14 - r_off) % 16
        got = run_agg_fwd(res, pre, (r_off, 4 * (r_off % 4), o_off))
        assert_bytes_equal(got, want, f"H={H} residual+{r_off} out+{o_off}")


@pytest.mark.parametrize("H", HS)
def test_every_phase_backward(H):
    T, n = 3, 4
    g, res, pre = backward_inputs(T, H, "ragged", 400 + H, n=n)
    want_gr, want_gp = oracle.aggregate_bwd(u16(g), u16(res), f32(pre), "bf16")
    for g_off in range(0, 16, 2):
        offs = (g_off, (g_off + 6) % 16, 4, (18 - g_off) % 16, 8)
        gr, gp = run_agg_bwd(g, res, pre, offs)
        assert_bytes_equal(gr, want_gr, f"grad_residual H={H} offsets={offs}")
        assert_bytes_equal(gp, want_gp, f"grad_pre H={H} offsets={offs}")


# rows of at least 256 chunks, every H mod 8
FIXED_HS = (2041, 2046, 2048, 2050, 2052, 2053, 4099, 7167)


@pytest.mark.parametrize("H", FIXED_HS)
def test_backward_residual_offsets_alike(H):
    """grad_residual at the residual's 16-byte offset (the compile-time window
    kernel for n = 4, BF16): every offset of g against every offset of the
    residual, over tokens whose rows step through the phases."""
    T, n = 5, 4
    g, res, pre = backward_inputs(T, H, "ragged", 800 + H, n=n)
    want_gr, want_gp = oracle.aggregate_bwd(u16(g), u16(res), f32(pre), "bf16")
    for g_off in range(0, 16, 2):
        for r_off in range(0, 16, 2):
            offs = (g_off, r_off, 4, r_off, 8)
            gr, gp = run_agg_bwd(g, res, pre, offs)
            assert_bytes_equal(gr, want_gr, f"grad_residual H={H} offsets={offs}")
            assert_bytes_equal(gp, want_gp, f"grad_pre H={H} offsets={offs}")


@pytest.mark.parametrize("dtype", (torch.bfloat16, torch.float16), ids=("bf16", "f16"))
@pytest.mark.parametrize("n", (1, 2, 8))
def test_streams_and_dtypes(n, dtype):
    T, H = 5, 4101
    g, res, pre = backward_inputs(T, H, "decode", 500 + n, n=n, dtype=dtype)
    name = DTYPE_NAME[dtype]
    want = oracle.aggregate_fwd(u16(res), f32(pre), name)
    want_gr, want_gp = oracle.aggregate_bwd(u16(g), u16(res), f32(pre), name)
    for offs in ((2, 4, 4, 10, 0), (14, 0, 0, 2, 4)):
        assert_bytes_equal(run_agg_fwd(res, pre, (offs[1], offs[2], offs[3])), want, f"fwd n={n} {offs}")
        gr, gp = run_agg_bwd(g, res, pre, offs)
        assert_bytes_equal(gr, want_gr, f"grad_residual n={n} {offs}")
        assert_bytes_equal(gp, want_gp, f"grad_pre n={n} {offs}")


def test_whole_buffer_ends():
    """One token (its rows are the whole buffers, so the first and last
    16-byte lines of each row are partly outside the buffer) at every phase."""
    H = 1001
    g, res, pre = backward_inputs(1, H, "normal", 600)
    want = oracle.aggregate_fwd(u16(res), f32(pre), "bf16")
    want_gr, want_gp = oracle.aggregate_bwd(u16(g), u16(res), f32(pre), "bf16")
    for off in range(2, 16, 2):
        assert_bytes_equal(run_agg_fwd(res, pre, (off, 0, off)), want, f"fwd +{off}")
        gr, gp = run_agg_bwd(g, res, pre, (off, off, 0, off, 0))
        assert_bytes_equal(gr, want_gr, f"grad_residual +{off}")
        assert_bytes_equal(gp, want_gp, f"grad_pre +{off}")


def test_large_odd_h_against_oracle():
    """T = 512, H = 7167 (every row at a different phase), the forward, the
    backward and the coefficients computed from the mix, through the tensor API."""
    from invariant_mhc_aggregate_gb300.inputs import coeff_inputs
    T, H = 512, 7167
    g, res, pre = backward_inputs(T, H, "normal", 700)
    gd, rd, pd = g.cuda(), res.cuda(), pre.cuda()
    out = binding.aggregate(rd, pd)
    assert binding.agg_fwd_path_raw(rd.data_ptr(), pd.data_ptr(), out.data_ptr(), T, 4, H) \
        == binding.MHC_PATH_SHIFT16
    gr, gp = binding.aggregate_backward(gd, rd, pd)
    assert_bytes_equal(u16(out), oracle.aggregate_fwd(u16(res), f32(pre)), "out")
    wgr, wgp = oracle.aggregate_bwd(u16(g), u16(res), f32(pre))
    assert_bytes_equal(u16(gr), wgr, "grad_residual")
    assert_bytes_equal(f32(gp), wgp, "grad_pre")
    mix, alpha, b = coeff_inputs(T, 4, "wide", 701)
    md, ad, bd = mix.cuda(), alpha.cuda(), b.cuda()
    a_np, b_np = np.float32(alpha.item()), b.numpy()
    assert_bytes_equal(u16(binding.aggregate_sigmoid(rd, md, ad, bd)),
                       oracle.aggregate_sigmoid_fwd(u16(res), f32(mix), a_np, b_np), "sigmoid out")
    sgr, sgz, sgm = binding.aggregate_sigmoid_backward(gd, rd, md, ad, bd)
    wgr, wgz, wgm = oracle.aggregate_sigmoid_bwd(u16(g), u16(res), f32(mix), a_np, b_np)
    assert_bytes_equal(u16(sgr), wgr, "sigmoid grad_residual")
    assert_bytes_equal(f32(sgz), wgz, "grad_z")
    assert_bytes_equal(f32(sgm), wgm, "grad_mix")


@pytest.mark.parametrize("H", (7167, 7166))
def test_realigned_backward_t4096_every_token(H):
    """The realigned backward at the benchmark's size (n = 4, BF16: the
    bulk-copy kernel, whose blocks each walk about 13 tokens through their
    ring): every output against the oracle, then 1- and 64-token calls, whose
    row blocks start and end part-way into 16-byte lines (the edge-token
    handling at every call)."""
    from test_configs_gpu import bwd_split, by_token_blocks, same_bytes
    T = 4096
    g, res, pre = backward_inputs(T, H, "normal", 900 + H)
    g_d, r_d, p_d = g.cuda(), res.cuda(), pre.cuda()
    gr, gp = binding.aggregate_backward(g_d, r_d, p_d)
    torch.cuda.synchronize()
    want_gr, want_gp = by_token_blocks(oracle.aggregate_bwd, u16(g), u16(res), f32(pre))
    assert_bytes_equal(u16(gr), want_gr, f"grad_residual H={H}")
    assert_bytes_equal(f32(gp), want_gp, f"grad_pre H={H}")
    for chunk in (1, 64):
        sgr, sgp = bwd_split(g_d, r_d, p_d, chunk)
        assert same_bytes(sgr, gr), f"grad_residual differs with {chunk}-token calls (H={H})"
        assert same_bytes(sgp, gp), f"grad_pre differs with {chunk}-token calls (H={H})"

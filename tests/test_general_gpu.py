"""The general form on the GPU: stream count n in {1, 2, 4, 8} and BF16 or
FP16 storage, against the CPU oracle byte for byte through the C ABI.

The pages fix n = 4 with BF16 ("Add batch-invariant h_aggregate kernel",
Summary); the balanced pairwise tree for other n and the FP16 variant are this
library's widening ("perf: fuse mHC coefficient backward epilogue", Testing
Done, exercises HC = {2,4,8} and FP16 alongside BF16).
"""

import numpy as np
import pytest
import torch

import oracle
import _pins
from _gpu import DTYPE_NAME, assert_bytes_equal, lib, run_agg_bwd, run_agg_fwd, sha, u16, f32
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.autograd import h_aggregate
from invariant_mhc_aggregate_gb300.inputs import backward_inputs, forward_inputs

pytestmark = pytest.mark.gpu

NS = (1, 2, 4, 8)
DTYPES = (torch.bfloat16, torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


def _ids(v):
    return DTYPE_NAME.get(v, str(v))


@pytest.mark.parametrize("dtype", DTYPES, ids=_ids)
@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("T,H", [(37, 7168), (5, 4096), (3, 4104), (2, 2050), (3, 1279), (129, 64)])
def test_forward_all_paths(n, dtype, T, H):
    res, pre = forward_inputs(T, H, "decode", 60 + n, n=n, dtype=dtype)
    want = oracle.aggregate_fwd(u16(res), f32(pre), DTYPE_NAME[dtype])
    for offsets in ((0, 0, 0), (16, 4, 0), (4, 0, 4), (2, 0, 2)):
        got = run_agg_fwd(res, pre, offsets)
        assert_bytes_equal(got, want, f"n={n} {DTYPE_NAME[dtype]} T={T} H={H} offsets={offsets}")


@pytest.mark.parametrize("dtype", DTYPES, ids=_ids)
@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("T,H", [(9, 7168), (3, 2048), (2, 4096), (2, 4112), (3, 1279), (1, 24)])
def test_backward_all_paths(n, dtype, T, H):
    g, res, pre = backward_inputs(T, H, "ragged", 70 + n, n=n, dtype=dtype)
    want_gr, want_gp = oracle.aggregate_bwd(u16(g), u16(res), f32(pre), DTYPE_NAME[dtype])
    for offsets in ((0, 0, 0, 0, 0), (16, 16, 4, 16, 4), (2, 0, 0, 0, 0)):
        gr, gp = run_agg_bwd(g, res, pre, offsets)
        what = f"n={n} {DTYPE_NAME[dtype]} T={T} H={H} offsets={offsets}"
        assert_bytes_equal(gr, want_gr, "grad_residual " + what)
        assert_bytes_equal(gp, want_gp, "grad_pre " + what)


def test_pages_op_is_n4_bf16():
    g, res, pre = backward_inputs(17, 7168, "normal", 81)
    gd, rd, pd = g.cuda(), res.cuda(), pre.cuda()
    a = binding.h_aggregate(rd, pd)
    b = binding.aggregate(rd, pd)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    gr1, gp1 = binding.h_aggregate_backward(gd, rd, pd)
    gr2, gp2 = binding.aggregate_backward(gd, rd, pd)
    assert torch.equal(gr1.view(torch.int16), gr2.view(torch.int16))
    assert torch.equal(gp1.view(torch.int32), gp2.view(torch.int32))


@pytest.mark.parametrize("offsets", [(0, 0, 0), (4, 0, 4), (2, 0, 2)])
def test_hc_worked_examples_on_gpu(offsets):
    rng = np.random.default_rng(61)
    for name, dtype, n, r, pre, expected in _pins._hc_cases():
        H = 16
        res = _pins.random_storage(rng, (3, n, H), dtype)
        pr = rng.random((3, n), dtype=np.float32)
        res[1, :, 5] = r
        pr[1] = pre
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
        rt = torch.from_numpy(res.view(np.int16).copy()).view(tdt)
        got = run_agg_fwd(rt, torch.from_numpy(pr), offsets)
        assert int(got[1, 5]) == expected, (name, offsets)
        assert_bytes_equal(got, oracle.aggregate_fwd(res, pr, dtype), name)


@pytest.mark.parametrize("n", (2, 8))
def test_f16_special_values(n):
    """binary16 overflow to infinity, subnormal results and signed zeros."""
    T, H = 8, 32
    rng = np.random.default_rng(62)
    res = _pins.random_f16(rng, (T, n, H), scale=100.0)
    res[0] = 0x8000                 # -0
    res[1, :, ::2] = 0x0001         # smallest subnormal
    res[2] = 0x7BFF                 # 65504
    pre = rng.random((T, n), dtype=np.float32)
    pre[2] = 4.0                    # overflow
    pre[3] = np.float32(2.0 ** -20) # subnormal results
    pre[4] = 0.0
    rt = torch.from_numpy(res.view(np.int16).copy()).view(torch.float16)
    for offsets in ((0, 0, 0), (2, 0, 2)):
        got = run_agg_fwd(rt, torch.from_numpy(pre), offsets)
        assert_bytes_equal(got, oracle.aggregate_fwd(res, pre, "f16"), f"f16 specials {offsets}")
    g = _pins.random_f16(rng, (T, H), scale=1000.0)
    g[5] = 0x0001
    gt = torch.from_numpy(g.view(np.int16).copy()).view(torch.float16)
    gr, gp = run_agg_bwd(gt, rt, torch.from_numpy(pre))
    want_gr, want_gp = oracle.aggregate_bwd(g, res, pre, "f16")
    assert_bytes_equal(gr, want_gr, "f16 grad_residual specials")
    assert_bytes_equal(gp, want_gp, "f16 grad_pre specials")


@pytest.mark.parametrize("n,dtype", [(8, torch.float16), (2, torch.bfloat16), (1, torch.float16)],
                         ids=["n8-f16", "n2-bf16", "n1-f16"])
def test_split_and_repeat_invariance(n, dtype):
    T, H = 256, 4096
    g, res, pre = backward_inputs(T, H, "normal", 90, n=n, dtype=dtype, device="cuda")
    out = binding.aggregate(res, pre)
    gr, gp = binding.aggregate_backward(g, res, pre)
    for _ in range(5):
        assert sha(binding.aggregate(res, pre)) == sha(out)
        gr2, gp2 = binding.aggregate_backward(g, res, pre)
        assert sha(gr2) == sha(gr) and sha(gp2) == sha(gp)
    for chunk in (1, 7, 64):
        o = torch.empty_like(out)
        gr3, gp3 = torch.empty_like(gr), torch.empty_like(gp)
        for t0 in range(0, T, chunk):
            sl = slice(t0, t0 + chunk)
            binding.mhc_aggregate_fwd(res[sl], pre[sl], o[sl])
            binding.mhc_aggregate_bwd(g[sl], res[sl], pre[sl], gr3[sl], gp3[sl])
        torch.cuda.synchronize()
        assert sha(o) == sha(out) and sha(gr3) == sha(gr) and sha(gp3) == sha(gp), chunk


@pytest.mark.parametrize("n,dtype", [(8, torch.float16), (2, torch.bfloat16)], ids=["n8-f16", "n2-bf16"])
def test_autograd_general(n, dtype):
    g, res, pre = backward_inputs(19, 2048, "normal", 95, n=n, dtype=dtype)
    r = res.cuda().requires_grad_(True)
    p = pre.cuda().requires_grad_(True)
    out = h_aggregate(r, p)
    out.backward(g.cuda())
    name = DTYPE_NAME[dtype]
    assert_bytes_equal(u16(out.detach()), oracle.aggregate_fwd(u16(res), f32(pre), name), "autograd fwd")
    want_gr, want_gp = oracle.aggregate_bwd(u16(g), u16(res), f32(pre), name)
    assert_bytes_equal(u16(r.grad), want_gr, "autograd grad_residual")
    assert_bytes_equal(f32(p.grad), want_gp, "autograd grad_pre")


def test_unsupported_stream_count_raises():
    res = torch.zeros((2, 3, 64), dtype=torch.bfloat16, device="cuda")
    pre = torch.zeros((2, 3), dtype=torch.float32, device="cuda")
    with pytest.raises(binding.MhcError):
        binding.aggregate(res, pre)

"""The pre coefficients computed from the mix, on the GPU, against the CPU
oracle byte for byte through the C ABI.

Source: "perf: fuse mHC coefficient backward epilogue" (Liger-Kernel pull
request 1402), Summary (pre sigmoid derivative, grad_mix, grad_b and alpha
gradients) and Risks and Limitations (fixed order of the grad_b / alpha
reductions).  The formulas and the binary32 sigmoid are this library's
reading and definition (see the oracle):
    z = RN(RN(alpha * mix) + b),  pre = sigmoid(z),  out = aggregate(residual, pre)
    grad_z = RN(grad_pre * sigmoid'(z)),  grad_mix = RN(alpha * grad_z)
    grad_b, grad_alpha: sums over tokens in ORDER-256.
"""

import numpy as np
import pytest
import torch

import oracle
import _pins
from _gpu import (DTYPE_CODE, DTYPE_NAME, DevBuf, assert_bytes_equal, expected_bwd_path,
                  expected_fwd_path, f32, lib, sha, stream_handle, u16)
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.autograd import h_aggregate_sigmoid
from invariant_mhc_aggregate_gb300.inputs import backward_inputs, coeff_inputs, forward_inputs

pytestmark = pytest.mark.gpu

NS = (1, 2, 4, 8)
DTYPES = (torch.bfloat16, torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


def _ids(v):
    return DTYPE_NAME.get(v, str(v))


def _scalar_buf(x: torch.Tensor, offset=0) -> DevBuf:
    return DevBuf.of(x.reshape(-1).to(torch.float32), offset)


def run_pre_sigmoid(mix, alpha, b, offsets=(0, 0, 0, 0)):
    T, n = mix.shape
    m = DevBuf.of(mix, offsets[0])
    a = _scalar_buf(alpha, offsets[1])
    bb = _scalar_buf(b, offsets[2])
    p = DevBuf(T * n * 4, offsets[3])
    st = binding.pre_sigmoid_raw(m.ptr, a.ptr, bb.ptr, p.ptr, T, n, stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    assert p.guards_ok(), "pre_sigmoid wrote outside pre"
    return p.get(np.float32, (T, n))


def run_sig_fwd(residual, mix, alpha, b, offsets=(0, 0, 0)):
    """offsets: residual, mix, out."""
    T, n, H = residual.shape
    r = DevBuf.of(residual, offsets[0])
    m = DevBuf.of(mix, offsets[1])
    a = _scalar_buf(alpha)
    bb = _scalar_buf(b)
    o = DevBuf(T * H * 2, offsets[2])
    assert binding.agg_fwd_path_raw(r.ptr, m.ptr, o.ptr, T, n, H) == expected_fwd_path(H, offsets)
    st = binding.agg_sigmoid_fwd_raw(r.ptr, m.ptr, a.ptr, bb.ptr, o.ptr, T, n, H,
                                     DTYPE_CODE[residual.dtype], stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    assert o.guards_ok(), "fused forward wrote outside out"
    return o.get(np.uint16, (T, H))


def run_sig_bwd(g, residual, mix, alpha, b, offsets=(0, 0, 0, 0, 0, 0)):
    """offsets: g, residual, mix, grad_residual, grad_z, grad_mix."""
    T, n, H = residual.shape
    gb = DevBuf.of(g, offsets[0])
    r = DevBuf.of(residual, offsets[1])
    m = DevBuf.of(mix, offsets[2])
    a = _scalar_buf(alpha)
    bb = _scalar_buf(b)
    gr = DevBuf(T * n * H * 2, offsets[3])
    gz = DevBuf(T * n * 4, offsets[4])
    gm = DevBuf(T * n * 4, offsets[5])
    assert binding.agg_bwd_path_raw(gb.ptr, r.ptr, m.ptr, gr.ptr, gz.ptr, T, n, H) == \
        expected_bwd_path(H, offsets[:2] + (0,) + offsets[3:4])
    st = binding.agg_sigmoid_bwd_raw(gb.ptr, r.ptr, m.ptr, a.ptr, bb.ptr, gr.ptr, gz.ptr, gm.ptr,
                                     T, n, H, DTYPE_CODE[residual.dtype], stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    assert gr.guards_ok() and gz.guards_ok() and gm.guards_ok(), "fused backward wrote outside"
    return gr.get(np.uint16, (T, n, H)), gz.get(np.float32, (T, n)), gm.get(np.float32, (T, n))


def run_param_grad(grad_z, mix, offsets=(0, 0, 0, 0)):
    T, n = grad_z.shape
    gz = DevBuf.of(grad_z, offsets[0]) if T else DevBuf(16, 0)
    m = DevBuf.of(mix, offsets[1]) if T else DevBuf(16, 0)
    gb = DevBuf(n * 4, offsets[2])
    ga = DevBuf(4, offsets[3])
    st = binding.sigmoid_param_grad_raw(gz.ptr, m.ptr, gb.ptr, ga.ptr, T, n, stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    assert gb.guards_ok() and ga.guards_ok(), "param grad wrote outside its outputs"
    return gb.get(np.float32, (n,)), ga.get(np.float32, (1,))[0]


def _np(alpha, b):
    return np.float32(alpha.reshape(-1)[0].item()), b.numpy().astype(np.float32)


# --------------------------------------------------------------------------
# the sigmoid itself
# --------------------------------------------------------------------------

def test_sigmoid_dense_sweep_bit_exact():
    """Every 61st binary32 value of [-128, 128] (about 35 million) as z: the
    device sigmoid equals the oracle's bit for bit."""
    zp = _pins.dense_floats(0x00000000, 0x43000000, 61)
    z = np.concatenate([zp, -zp]).astype(np.float32)
    T = len(z)
    mix = torch.from_numpy(z.reshape(T, 1))
    got = run_pre_sigmoid(mix, torch.ones(1), torch.zeros(1))
    want, _ = oracle.default().sigmoid32(z + np.float32(0.0))
    assert_bytes_equal(got.reshape(-1), want, "sigmoid sweep")


def test_sigmoid_special_values():
    z = np.float32([0.0, -0.0, np.inf, -np.inf, 100.0, -100.0, 20.0, -20.0, 1e-30, -1e-30,
                    3.4e38, -3.4e38, 88.7, -88.7, 103.9, -103.9, 104.5, -104.5])
    mix = torch.from_numpy(z.reshape(-1, 1))
    got = run_pre_sigmoid(mix, torch.ones(1), torch.zeros(1))
    want, _ = oracle.default().sigmoid32(z + np.float32(0.0))
    assert_bytes_equal(got.reshape(-1), want, "special z")
    nan = run_pre_sigmoid(torch.tensor([[float("nan")]]), torch.ones(1), torch.zeros(1))
    assert np.isnan(nan).all()


def test_sigmoid_close_to_cuda_sigmoid():
    """Against CUDA's own sigmoid (torch.sigmoid on the device) where neither
    underflows: within 8 binary32 ulps (this library's is within 2.5 of the
    exact value)."""
    rng = np.random.default_rng(7)
    z = np.concatenate([rng.uniform(-80, 80, 200000), rng.standard_normal(200000) * 3]).astype(np.float32)
    mix = torch.from_numpy(z.reshape(-1, 1))
    got = run_pre_sigmoid(mix, torch.ones(1), torch.zeros(1)).reshape(-1).astype(np.float64)
    ref = torch.sigmoid(mix.cuda()).cpu().numpy().reshape(-1).astype(np.float64)
    err = np.abs(got - ref) / _pins.f32_ulp(ref)
    assert err.max() <= 8.0, f"max {err.max():.2f} ulp at z={z[err.argmax()]}"


@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("recipe", ("normal", "wide"))
def test_pre_sigmoid_matches_oracle(n, recipe):
    for T in (1, 37, 4099):
        mix, alpha, b = coeff_inputs(T, n, recipe, 100 + n)
        want = oracle.pre_sigmoid(f32(mix), *_np(alpha, b))
        for offsets in ((0, 0, 0, 0), (4, 4, 8, 4)):
            got = run_pre_sigmoid(mix, alpha, b, offsets)
            assert_bytes_equal(got, want, f"pre n={n} {recipe} T={T} {offsets}")


# --------------------------------------------------------------------------
# fused forward and backward
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES, ids=_ids)
@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("T,H", [(37, 7168), (3, 4104), (2, 2050), (3, 1279), (129, 64)])
def test_fused_forward_all_paths(n, dtype, T, H):
    res, _ = forward_inputs(T, H, "decode", 110 + n, n=n, dtype=dtype)
    mix, alpha, b = coeff_inputs(T, n, "wide", 120 + n)
    want = oracle.aggregate_sigmoid_fwd(u16(res), f32(mix), *_np(alpha, b), DTYPE_NAME[dtype])
    for offsets in ((0, 0, 0), (16, 4, 0), (4, 8, 4), (2, 0, 2)):
        got = run_sig_fwd(res, mix, alpha, b, offsets)
        assert_bytes_equal(got, want, f"n={n} {DTYPE_NAME[dtype]} T={T} H={H} {offsets}")


@pytest.mark.parametrize("dtype", DTYPES, ids=_ids)
@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("T,H", [(9, 7168), (3, 2048), (2, 4112), (3, 1279), (1, 24)])
def test_fused_backward_all_paths(n, dtype, T, H):
    g, res, _ = backward_inputs(T, H, "normal", 130 + n, n=n, dtype=dtype)
    mix, alpha, b = coeff_inputs(T, n, "wide", 140 + n)
    want = oracle.aggregate_sigmoid_bwd(u16(g), u16(res), f32(mix), *_np(alpha, b),
                                        DTYPE_NAME[dtype])
    for offsets in ((0, 0, 0, 0, 0, 0), (16, 16, 4, 16, 4, 8), (2, 0, 0, 0, 0, 0)):
        got = run_sig_bwd(g, res, mix, alpha, b, offsets)
        what = f"n={n} {DTYPE_NAME[dtype]} T={T} H={H} {offsets}"
        for name, x, y in zip(("grad_residual", "grad_z", "grad_mix"), got, want):
            assert_bytes_equal(x, y, f"{name} {what}")


@pytest.mark.parametrize("n", (2, 4))
def test_fused_equals_composition_on_gpu(n):
    """The fused calls give the bytes of pre_sigmoid followed by the plain
    aggregate calls (and grad_residual of the plain backward)."""
    T, H = 65, 7168
    g, res, _ = backward_inputs(T, H, "normal", 150, n=n)
    mix, alpha, b = coeff_inputs(T, n, "normal", 151)
    gd, rd, md, ad, bd = (x.cuda() for x in (g, res, mix, alpha, b))
    pre = binding.pre_sigmoid(md, ad, bd)
    assert torch.equal(binding.aggregate_sigmoid(rd, md, ad, bd).view(torch.int16),
                       binding.aggregate(rd, pre).view(torch.int16))
    gr1, gz, gm = binding.aggregate_sigmoid_backward(gd, rd, md, ad, bd)
    gr2, gp = binding.aggregate_backward(gd, rd, pre)
    assert torch.equal(gr1.view(torch.int16), gr2.view(torch.int16))
    # grad_mix = RN(alpha * grad_z), a property of the two outputs
    assert np.array_equal(f32(gm).view(np.uint32), _pins.f32_bits(f32(ad)[0] * f32(gz)))
    # where sigmoid'(z) = 1/4 exactly (z = 0), grad_z = grad_pre / 4 exactly
    z0 = torch.zeros_like(md)
    _, gz0, _ = binding.aggregate_sigmoid_backward(gd, rd, z0, ad, torch.zeros_like(bd))
    _, gp0 = binding.aggregate_backward(gd, rd, torch.full_like(md, 0.5))
    assert torch.equal(gz0, gp0 / 4)


def test_fused_full_size_against_oracle():
    """T = 4096, H = 7168, n = 4, BF16 (the backward benchmark's shape), the
    whole output against the oracle, in the launch configuration the benchmark
    uses (torch allocations, the current stream)."""
    T, H = 4096, 7168
    g, res, _ = backward_inputs(T, H, "normal", 4)
    mix, alpha, b = coeff_inputs(T, 4, "normal", 5)
    gd, rd, md, ad, bd = (x.cuda() for x in (g, res, mix, alpha, b))
    out = binding.aggregate_sigmoid(rd, md, ad, bd)
    gr, gz, gm = binding.aggregate_sigmoid_backward(gd, rd, md, ad, bd)
    gb, ga = binding.sigmoid_param_grad(gz, md)
    torch.cuda.synchronize()
    o = oracle.default()
    a_np, b_np = _np(alpha, b)
    assert_bytes_equal(u16(out), o.aggregate_sigmoid_fwd(u16(res), f32(mix), a_np, b_np), "out")
    wgr, wgz, wgm = o.aggregate_sigmoid_bwd(u16(g), u16(res), f32(mix), a_np, b_np)
    assert_bytes_equal(u16(gr), wgr, "grad_residual")
    assert_bytes_equal(f32(gz), wgz, "grad_z")
    assert_bytes_equal(f32(gm), wgm, "grad_mix")
    wgb, wga = o.sigmoid_param_grad(wgz, f32(mix))
    assert_bytes_equal(f32(gb), wgb, "grad_b")
    assert f32(ga).view(np.uint32)[0] == np.float32(wga).view(np.uint32)


@pytest.mark.parametrize("n", (1, 4, 8))
def test_fused_batch_split_invariance(n):
    T, H = 64, 4096
    g, res, _ = backward_inputs(T, H, "normal", 160, n=n)
    mix, alpha, b = coeff_inputs(T, n, "wide", 161)
    gd, rd, md, ad, bd = (x.cuda() for x in (g, res, mix, alpha, b))
    full = binding.aggregate_sigmoid(rd, md, ad, bd)
    fgr, fgz, fgm = binding.aggregate_sigmoid_backward(gd, rd, md, ad, bd)
    for chunk in (1, 7, 64):
        for t0 in range(0, T, chunk):
            t1 = min(T, t0 + chunk)
            part = binding.aggregate_sigmoid(rd[t0:t1].contiguous(), md[t0:t1].contiguous(), ad, bd)
            assert torch.equal(part.view(torch.int16), full[t0:t1].view(torch.int16)), (chunk, t0)
            pgr, pgz, pgm = binding.aggregate_sigmoid_backward(
                gd[t0:t1].contiguous(), rd[t0:t1].contiguous(), md[t0:t1].contiguous(), ad, bd)
            assert torch.equal(pgr.view(torch.int16), fgr[t0:t1].view(torch.int16))
            assert torch.equal(pgz.view(torch.int32), fgz[t0:t1].view(torch.int32))
            assert torch.equal(pgm.view(torch.int32), fgm[t0:t1].view(torch.int32))


def test_fused_repeat_calls_identical():
    T, H = 300, 7168
    g, res, _ = backward_inputs(T, H, "normal", 170)
    mix, alpha, b = coeff_inputs(T, 4, "normal", 171)
    gd, rd, md, ad, bd = (x.cuda() for x in (g, res, mix, alpha, b))
    ref = None
    for _ in range(20):
        out = binding.aggregate_sigmoid(rd, md, ad, bd)
        gr, gz, gm = binding.aggregate_sigmoid_backward(gd, rd, md, ad, bd)
        gb, ga = binding.sigmoid_param_grad(gz, md)
        h = tuple(sha(x) for x in (out, gr, gz, gm, gb, ga))
        assert ref is None or h == ref
        ref = h


# --------------------------------------------------------------------------
# the parameter gradients
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", NS)
def test_param_grad_matches_oracle(n):
    rng = np.random.default_rng(180 + n)
    for T in (1, 5, 8, 9, 300, 2047, 2048, 2049, 4096, 8191, 65536, 70001):
        gz = rng.standard_normal((T, n)).astype(np.float32)
        mix = (rng.standard_normal((T, n)) * 4).astype(np.float32)
        want_b, want_a = oracle.sigmoid_param_grad(gz, mix)
        for offsets in ((0, 0, 0, 0), (4, 4, 4, 4)):
            gb, ga = run_param_grad(torch.from_numpy(gz), torch.from_numpy(mix), offsets)
            assert_bytes_equal(gb, want_b, f"grad_b n={n} T={T} {offsets}")
            assert np.float32(ga).view(np.uint32) == np.float32(want_a).view(np.uint32), (n, T)


def test_param_grad_zero_tokens_writes_zeros():
    gb, ga = run_param_grad(torch.zeros((0, 4)), torch.zeros((0, 4)))
    assert np.all(gb.view(np.uint32) == 0) and np.float32(ga).view(np.uint32) == 0


def test_param_grad_order_golden_on_gpu():
    """The ORDER-256 golden cases with tokens in place of h (as in the oracle pins)."""
    vals_of = {0x3F80: 1.0, 0x3380: 2.0 ** -24, 0x8000: -0.0}
    for name, H, k, _c, positions, expected in _pins.golden_rows("grad_pre_order_cases.txt"):
        T, k = int(H), int(k)
        col = np.zeros(T, dtype=np.float32)
        for item in positions.split(","):
            pos, v = item.split(":")
            if pos == "*":
                col[:] = vals_of[int(v, 16)]
            else:
                col[int(pos)] = vals_of[int(v, 16)]
        gz = np.zeros((T, 4), dtype=np.float32)
        gz[:, k] = col
        gb, _ = run_param_grad(torch.from_numpy(gz), torch.ones((T, 4)))
        assert int(gb.view(np.uint32)[k]) == int(expected, 16), name
        _, ga = run_param_grad(torch.from_numpy(col[:, None].copy()), torch.ones((T, 1)))
        assert int(np.float32(ga).view(np.uint32)) == int(expected, 16), name


# --------------------------------------------------------------------------
# autograd and graphs
# --------------------------------------------------------------------------

def test_autograd_gradients_match_oracle():
    T, H, n = 33, 2048, 4
    g, res, _ = backward_inputs(T, H, "normal", 190)
    mix, alpha, b = coeff_inputs(T, n, "normal", 191)
    r = res.cuda().requires_grad_(True)
    m = mix.cuda().requires_grad_(True)
    a = alpha.reshape(()).cuda().requires_grad_(True)
    bb = b.cuda().requires_grad_(True)
    out = h_aggregate_sigmoid(r, m, a, bb)
    out.backward(g.cuda())
    o = oracle.default()
    a_np, b_np = _np(alpha, b)
    assert_bytes_equal(u16(out.detach()), o.aggregate_sigmoid_fwd(u16(res), f32(mix), a_np, b_np), "out")
    wgr, wgz, wgm = o.aggregate_sigmoid_bwd(u16(g), u16(res), f32(mix), a_np, b_np)
    wgb, wga = o.sigmoid_param_grad(wgz, f32(mix))
    assert_bytes_equal(u16(r.grad), wgr, "residual.grad")
    assert_bytes_equal(f32(m.grad), wgm, "mix.grad")
    assert_bytes_equal(f32(bb.grad), wgb, "b.grad")
    assert a.grad.shape == () and f32(a.grad).view(np.uint32) == np.float32(wga).view(np.uint32)


def test_autograd_training_converges():
    """Fit mix, alpha and b so that the fused aggregate reproduces a target
    built from different coefficients: the loss must fall by 10x."""
    torch.manual_seed(0)
    T, H, n = 64, 512, 4
    res = torch.randn(T, n, H, device="cuda").to(torch.bfloat16)
    target_pre = torch.rand(T, n, device="cuda") * 0.8 + 0.1
    target = binding.aggregate(res, target_pre).float()
    m = torch.zeros(T, n, device="cuda", requires_grad=True)
    a = torch.ones((), device="cuda", requires_grad=True)
    bb = torch.zeros(n, device="cuda", requires_grad=True)
    opt = torch.optim.Adam([m, a, bb], lr=0.05)
    first = None
    for _ in range(300):
        opt.zero_grad()
        out = h_aggregate_sigmoid(res, m, a, bb)
        loss = (out.float() - target).square().mean()
        if first is None:
            first = float(loss)
        loss.backward()
        opt.step()
    assert float(loss) < first / 10, (first, float(loss))


def test_fused_calls_capture_in_a_graph():
    T, H, n = 128, 4096, 4
    g, res, _ = backward_inputs(T, H, "normal", 200)
    mix, alpha, b = coeff_inputs(T, n, "normal", 201)
    gd, rd, md, ad, bd = (x.cuda() for x in (g, res, mix, alpha, b))
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    gr = torch.empty(T, n, H, dtype=torch.bfloat16, device="cuda")
    gz = torch.empty(T, n, device="cuda")
    gm = torch.empty(T, n, device="cuda")
    gb = torch.empty(n, device="cuda")
    ga = torch.empty(1, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        binding.mhc_aggregate_sigmoid_fwd(rd, md, ad, bd, out)   # warm-up outside capture
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=s):
            binding.mhc_aggregate_sigmoid_fwd(rd, md, ad, bd, out)
            binding.mhc_aggregate_sigmoid_bwd(gd, rd, md, ad, bd, gr, gz, gm)
            binding.mhc_sigmoid_param_grad(gz, md, gb, ga)
    for x in (out, gr, gz, gm, gb, ga):
        x.zero_()
    graph.replay()
    torch.cuda.synchronize()
    e_out = binding.aggregate_sigmoid(rd, md, ad, bd)
    e_gr, e_gz, e_gm = binding.aggregate_sigmoid_backward(gd, rd, md, ad, bd)
    e_gb, e_ga = binding.sigmoid_param_grad(e_gz, md)
    for x, y in ((out, e_out), (gr, e_gr), (gz, e_gz), (gm, e_gm), (gb, e_gb), (ga, e_ga)):
        assert sha(x) == sha(y)


def test_four_way_report_with_sigmoid_coefficients():
    """The reviewer's four checks for the aggregate with pre computed from the
    mix: forward and gradient accuracy against FP64 (with bounds from the
    binary32 steps), forward and gradient invariance under a batch split and
    repeats."""
    T, H, n = 128, 7168, 4
    g, res, _ = backward_inputs(T, H, "normal", 210)
    mix, alpha, b = coeff_inputs(T, n, "normal", 211)
    gd, rd, md, ad, bd = (x.cuda() for x in (g, res, mix, alpha, b))
    out = binding.aggregate_sigmoid(rd, md, ad, bd)
    gr, gz, gm = binding.aggregate_sigmoid_backward(gd, rd, md, ad, bd)
    gb, ga = binding.sigmoid_param_grad(gz, md)
    torch.cuda.synchronize()
    U = 2.0 ** -24
    a64 = float(alpha.item())
    z64 = a64 * f32(mix).astype(np.float64) + f32(b).astype(np.float64)[None, :]
    s64 = _pins.sigmoid64(z64)
    ds64 = s64 * _pins.sigmoid64(-z64)
    dz = 2.02 * U * (np.abs(a64 * f32(mix).astype(np.float64)) + np.abs(f32(b)).astype(np.float64)[None, :])
    rw = _pins.bf16_widen(u16(res)).astype(np.float64)
    gw = _pins.bf16_widen(u16(g)).astype(np.float64)
    # forward: exact sum of sigmoid(z_k) * r_k; bound = half a BF16 ulp + the
    # tree's rounding + each pre_k's error (2.5 ulp of the sigmoid, plus the
    # rounding of z carried through the slope)
    exact = np.einsum("tk,tkh->th", s64, rw)
    pre_err = 2.5 * _pins.f32_ulp(s64) + ds64 * dz
    o64 = _pins.bf16_widen(u16(out)).astype(np.float64)
    bound = (0.5 * _pins.bf16_ulp(o64) + 3.01 * U * np.einsum("tk,tkh->th", s64, np.abs(rw))
             + np.einsum("tk,tkh->th", pre_err, np.abs(rw)))
    fwd_ratio = float(np.max(np.abs(o64 - exact) / bound))
    # gradients: grad_mix = alpha * sigmoid'(z) * sum_h g r, relative to the
    # magnitude sum |alpha sigmoid' g r| (cancellation makes a plain relative
    # error meaningless), within 1e-3
    q = np.einsum("th,tkh->tk", gw, rw)
    qa = np.einsum("th,tkh->tk", np.abs(gw), np.abs(rw))
    exact_gm = a64 * ds64 * q
    scale = np.maximum(np.abs(exact_gm), np.abs(a64) * ds64 * qa)
    gm_err = float(np.max(np.abs(f32(gm).astype(np.float64) - exact_gm) / scale))
    exact_gz = ds64 * q
    gb_exact = exact_gz.sum(axis=0)
    gb_scale = np.abs(exact_gz).sum(axis=0) + 1e-30
    gb_err = float(np.max(np.abs(f32(gb).astype(np.float64) - gb_exact) / gb_scale))
    ga_exact = float((exact_gz * f32(mix).astype(np.float64)).sum())
    ga_err = abs(float(ga.item()) - ga_exact) / float(np.abs(exact_gz * f32(mix)).sum())
    # invariance: the batch split into halves, and a repeat
    h0 = T // 2
    part0 = binding.aggregate_sigmoid(rd[:h0].contiguous(), md[:h0].contiguous(), ad, bd)
    p_gr, p_gz, p_gm = binding.aggregate_sigmoid_backward(gd[h0:].contiguous(), rd[h0:].contiguous(),
                                                          md[h0:].contiguous(), ad, bd)
    fwd_inv = torch.equal(part0.view(torch.int16), out[:h0].view(torch.int16)) and \
        sha(binding.aggregate_sigmoid(rd, md, ad, bd)) == sha(out)
    grad_inv = torch.equal(p_gr.view(torch.int16), gr[h0:].view(torch.int16)) and \
        torch.equal(p_gz.view(torch.int32), gz[h0:].view(torch.int32)) and \
        torch.equal(p_gm.view(torch.int32), gm[h0:].view(torch.int32))
    report = {"forward_accuracy (error / bound)": fwd_ratio, "gradient_accuracy grad_mix": gm_err,
              "gradient_accuracy grad_b": gb_err, "gradient_accuracy grad_alpha": ga_err,
              "forward_invariance": fwd_inv, "gradient_invariance": grad_inv}
    print(report)
    assert fwd_ratio <= 1.0 and gm_err <= 1e-3 and gb_err <= 1e-3 and ga_err <= 1e-3, report
    assert fwd_inv and grad_inv, report

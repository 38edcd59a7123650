"""The mHC post on the GPU, against the CPU oracle byte for byte through the C ABI.

Source: "Add batch-invariant h_aggregate kernel", Summary, names the stage
("MHC Post"); "perf: fuse mHC coefficient backward epilogue", Summary, names
its post and residual-mixing coefficients.  The formula is the library's
reading (the hyper-connection update, see the oracle):
    out[t,k,h]      = cvt(tree_n(res[t,k,j] * x[t,j,h]) + post[t,k] * y[t,h])
    grad_x[t,j,h]   = cvt(tree_n over k of res[t,k,j] * g[t,k,h])
    grad_y[t,h]     = cvt(tree_n over k of post[t,k] * g[t,k,h])
    grad_res, grad_post: sums over h in ORDER-256.
"""

import numpy as np
import pytest
import torch

import oracle
from _gpu import (DTYPE_CODE, DTYPE_NAME, DevBuf, _align_of, assert_bytes_equal, f32, lib, sha,
                  stream_handle, u16)
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.autograd import mhc_post
from invariant_mhc_aggregate_gb300.inputs import post_inputs

pytestmark = pytest.mark.gpu

NS = (1, 2, 4, 8)
DTYPES = (torch.bfloat16, torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


def _ids(v):
    return DTYPE_NAME.get(v, str(v))


def expected_post_fwd_path(H, offsets):
    """offsets: x, y, post, res, out."""
    a = min(_align_of(offsets[0]), _align_of(offsets[1]), _align_of(offsets[4]))
    if H % 8 == 0 and a >= 16:
        return binding.MHC_PATH_VEC16
    return binding.MHC_PATH_ELEMENT


def expected_post_bwd_path(H, offsets):
    """offsets: g, x, y, post, res, grad_x, grad_y, grad_post, grad_res."""
    a = min(_align_of(offsets[i]) for i in (0, 1, 2, 5, 6))
    if H % 8 == 0 and a >= 16:
        return binding.MHC_PATH_VEC16
    return binding.MHC_PATH_ELEMENT


def run_post_fwd(x, y, post, res, offsets=(0,) * 5):
    T, n, H = x.shape
    bx, by = DevBuf.of(x, offsets[0]), DevBuf.of(y, offsets[1])
    bp, br = DevBuf.of(post, offsets[2]), DevBuf.of(res, offsets[3])
    bo = DevBuf(T * n * H * 2, offsets[4])
    assert binding.post_fwd_path_raw(bx.ptr, by.ptr, bp.ptr, br.ptr, bo.ptr, T, n, H) == \
        expected_post_fwd_path(H, offsets)
    st = binding.post_fwd_raw(bx.ptr, by.ptr, bp.ptr, br.ptr, bo.ptr, T, n, H, DTYPE_CODE[x.dtype],
                              stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    assert bo.guards_ok(), "post forward wrote outside out"
    return bo.get(np.uint16, (T, n, H))


def run_post_bwd(g, x, y, post, res, offsets=(0,) * 9):
    T, n, H = x.shape
    ins = [DevBuf.of(t, o) for t, o in zip((g, x, y, post, res), offsets[:5])]
    outs = [DevBuf(T * n * H * 2, offsets[5]), DevBuf(T * H * 2, offsets[6]),
            DevBuf(T * n * 4, offsets[7]), DevBuf(T * n * n * 4, offsets[8])]
    ptrs = [b.ptr for b in ins + outs]
    assert binding.post_bwd_path_raw(*ptrs, T, n, H) == expected_post_bwd_path(H, offsets)
    st = binding.post_bwd_raw(*ptrs, T, n, H, DTYPE_CODE[x.dtype], stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    assert all(b.guards_ok() for b in outs), "post backward wrote outside its outputs"
    return (outs[0].get(np.uint16, (T, n, H)), outs[1].get(np.uint16, (T, H)),
            outs[2].get(np.float32, (T, n)), outs[3].get(np.float32, (T, n, n)))


# (T, H, offsets of x, y, post, res, out): each forward path, rows spanning
# several blocks and ragged tails, tokens straddling blocks of the flat grid
FWD_CASES = [
    (5, 4096, (0, 0, 0, 0, 0)),        # 16-byte vectors
    (3, 7168, (0, 0, 4, 4, 0)),        # a block spans two tokens
    (7, 4104, (0, 0, 0, 0, 0)),        # H % 16 == 8
    (4, 4096, (16, 0, 0, 0, 0)),       # x only 16-byte aligned
    (3, 4100, (0, 0, 0, 0, 0)),        # H % 8 != 0: 2-byte path
    (2, 1279, (0, 2, 0, 0, 6)),        # odd H, 2-byte aligned buffers
    (9, 8, (0, 0, 0, 0, 0)),           # one 16-byte vector a row
    (3, 1, (0, 0, 0, 0, 0)),           # one value a row
    (1, 2048 + 16, (0, 0, 0, 0, 0)),   # a single token
    (5, 1024, (0, 0, 0, 0, 0)),        # 128 vectors a row
    (5, 512, (0, 0, 0, 0, 0)),         # 64 vectors a row: n = 8's split forward from here on
    (5, 504, (0, 0, 0, 0, 0)),         # 63 vectors a row: n = 8's one-thread-per-vector forward
    (37, 520, (0, 0, 0, 0, 0)),        # 65 vectors a row: split blocks span two tokens
]


@pytest.mark.parametrize("dtype", DTYPES, ids=_ids)
@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("T,H,offsets", FWD_CASES)
def test_post_fwd_all_paths(T, H, offsets, n, dtype):
    x, y, post, res = post_inputs(T, H, n, "normal", 300 + T + H, dtype=dtype)
    got = run_post_fwd(x, y, post, res, offsets)
    want = oracle.post_fwd(u16(x), u16(y), f32(post), f32(res), DTYPE_NAME[dtype])
    assert_bytes_equal(got, want, "out")


# (T, H, offsets of g, x, y, post, res, grad_x, grad_y, grad_post, grad_res)
BWD_CASES = [
    (5, 4096, (0,) * 9),                               # 16-byte chunks, 2 a lane
    (3, 7168, (0, 0, 0, 4, 4, 0, 0, 4, 4)),            # 3.5 chunks a lane
    (7, 4104, (0,) * 9),
    (2, 1024, (0,) * 9),                               # fewer chunks than lanes
    (4, 4096, (0, 0, 0, 0, 0, 0, 8, 0, 0)),            # grad_y off 16 bytes: 2-byte path
    (3, 4100, (0,) * 9),                               # ragged last chunk
    (2, 1279, (2, 0, 6, 0, 0, 2, 0, 0, 0)),
    (9, 8, (0,) * 9),
    (3, 1, (0,) * 9),
    (1, 2048 * 8 + 8, (0,) * 9),                       # long row: 8+ chunks a lane
    (3, 8 * (256 + 37), (0,) * 9),                     # last segment ends inside a warp's lanes
    # n = 8 tensor maps group a row in the widest power of two up to 256
    # that divides H: 16, 32, 64 and 128 values here (256 and 8 above)
    (3, 4112, (0,) * 9),
    (3, 2080, (0,) * 9),
    (3, 2112, (0,) * 9),
    (3, 2176, (0,) * 9),
]


@pytest.mark.parametrize("dtype", DTYPES, ids=_ids)
@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("T,H,offsets", BWD_CASES)
def test_post_bwd_all_paths(T, H, offsets, n, dtype):
    x, y, post, res, g = post_inputs(T, H, n, "normal", 400 + T + H, dtype=dtype, with_grad=True)
    got = run_post_bwd(g, x, y, post, res, offsets)
    want = oracle.post_bwd(u16(g), u16(x), u16(y), f32(post), f32(res), DTYPE_NAME[dtype])
    for a, b, what in zip(got, want, ("grad_x", "grad_y", "grad_post", "grad_res")):
        assert_bytes_equal(a, b, what)


@pytest.mark.parametrize("n", NS)
def test_post_ragged_recipe(n):
    """Identity mixing rows and zero post coefficients."""
    T, H = 40, 2048
    x, y, post, res, g = post_inputs(T, H, n, "ragged", 500 + n, with_grad=True)
    xd, yd, pd, rd, gd = (t.cuda() for t in (x, y, post, res, g))
    out = binding.post(xd, yd, pd, rd)
    gx, gy, gp, gr = binding.post_backward(gd, xd, yd, pd, rd)
    torch.cuda.synchronize()
    o = oracle.default()
    assert_bytes_equal(u16(out), o.post_fwd(u16(x), u16(y), f32(post), f32(res)), "out")
    want = o.post_bwd(u16(g), u16(x), u16(y), f32(post), f32(res))
    for a, b, what in zip((u16(gx), u16(gy), f32(gp), f32(gr)), want,
                          ("grad_x", "grad_y", "grad_post", "grad_res")):
        assert_bytes_equal(a, b, what)


def test_post_full_size_against_oracle():
    """T = 4096, H = 7168, n = 4, BF16 (the benchmark's shape), every output
    against the oracle, in the launch configuration the benchmark uses (torch
    allocations, the current stream)."""
    T, H, n = 4096, 7168, 4
    x, y, post, res, g = post_inputs(T, H, n, "normal", 6, with_grad=True)
    xd, yd, pd, rd, gd = (t.cuda() for t in (x, y, post, res, g))
    out = binding.post(xd, yd, pd, rd)
    gx, gy, gp, gr = binding.post_backward(gd, xd, yd, pd, rd)
    torch.cuda.synchronize()
    o = oracle.default()
    assert_bytes_equal(u16(out), o.post_fwd(u16(x), u16(y), f32(post), f32(res)), "out")
    want = o.post_bwd(u16(g), u16(x), u16(y), f32(post), f32(res))
    for a, b, what in zip((u16(gx), u16(gy), f32(gp), f32(gr)), want,
                          ("grad_x", "grad_y", "grad_post", "grad_res")):
        assert_bytes_equal(a, b, what)


@pytest.mark.parametrize("n", (1, 4, 8))
def test_post_batch_split_invariance(n):
    """Every token's outputs are the same bytes whatever batch it is run in."""
    T, H = 64, 4096
    x, y, post, res, g = post_inputs(T, H, n, "normal", 600 + n, with_grad=True)
    xd, yd, pd, rd, gd = (t.cuda() for t in (x, y, post, res, g))
    full = binding.post(xd, yd, pd, rd)
    fgrads = binding.post_backward(gd, xd, yd, pd, rd)
    for chunk in (1, 7, 64):
        for t0 in range(0, T, chunk):
            sl = slice(t0, min(T, t0 + chunk))
            args = [t[sl].contiguous() for t in (xd, yd, pd, rd)]
            part = binding.post(*args)
            assert sha(part) == sha(full[sl]), (chunk, t0)
            pgrads = binding.post_backward(gd[sl].contiguous(), *args)
            for p, f in zip(pgrads, fgrads):
                assert sha(p) == sha(f[sl]), (chunk, t0)


@pytest.mark.parametrize("n", (4, 8))
def test_post_repeat_calls_identical(n):
    """Repeated calls on the same inputs give the same bytes (the bulk-copy
    rings, the partner exchange and the folds hold no state between calls)."""
    T, H = 512, 7168
    x, y, post, res, g = (t.cuda() for t in post_inputs(T, H, n, "normal", 700, with_grad=True))
    first = [sha(binding.post(x, y, post, res))] + [sha(t) for t in binding.post_backward(g, x, y, post, res)]
    for _ in range(10):
        again = [sha(binding.post(x, y, post, res))] + [sha(t) for t in binding.post_backward(g, x, y, post, res)]
        assert again == first


def test_post_autograd_gradients_match_oracle():
    T, H, n = 2 * 17, 2048, 4
    x, y, post, res, g = post_inputs(T, H, n, "normal", 800, with_grad=True)
    xd = x.cuda().reshape(2, 17, n, H).requires_grad_(True)
    yd = y.cuda().reshape(2, 17, H).requires_grad_(True)
    pd = post.cuda().reshape(2, 17, n).requires_grad_(True)
    rd = res.cuda().reshape(2, 17, n, n).requires_grad_(True)
    out = mhc_post(xd, yd, pd, rd)
    assert out.shape == (2, 17, n, H)
    out.backward(g.cuda().reshape(2, 17, n, H))
    o = oracle.default()
    assert_bytes_equal(u16(out.detach().reshape(T, n, H)),
                       o.post_fwd(u16(x), u16(y), f32(post), f32(res)), "out")
    wgx, wgy, wgp, wgr = o.post_bwd(u16(g), u16(x), u16(y), f32(post), f32(res))
    assert_bytes_equal(u16(xd.grad.reshape(T, n, H)), wgx, "x.grad")
    assert_bytes_equal(u16(yd.grad.reshape(T, H)), wgy, "y.grad")
    assert_bytes_equal(f32(pd.grad.reshape(T, n)), wgp, "post.grad")
    assert_bytes_equal(f32(rd.grad.reshape(T, n, n)), wgr, "res.grad")


def test_post_identity_on_gpu():
    """res = I and post = 0 give out = x exactly; post = 1 and x = 0 give
    out = y exactly (the oracle's special cases, through the kernels)."""
    T, H, n = 16, 4096, 4
    x, y, post, res = post_inputs(T, H, n, "normal", 900)
    xd, yd = x.cuda(), y.cuda()
    eye = torch.eye(n, device="cuda").expand(T, n, n).contiguous()
    out = binding.post(xd, yd, torch.zeros(T, n, device="cuda"), eye)
    assert sha(out) == sha(xd)
    out = binding.post(torch.zeros_like(xd), yd, torch.ones(T, n, device="cuda"), eye)
    assert sha(out) == sha(yd[:, None, :].expand(T, n, H).contiguous())


def test_post_calls_capture_in_a_graph():
    T, H, n = 128, 4096, 4
    x, y, post, res, g = (t.cuda() for t in post_inputs(T, H, n, "normal", 950, with_grad=True))
    out = torch.empty_like(x)
    gx, gy = torch.empty_like(x), torch.empty_like(y)
    gp, gr = torch.empty_like(post), torch.empty_like(res)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        binding.mhc_post_fwd(x, y, post, res, out)
        torch.cuda.synchronize()
        with torch.cuda.graph(graph, stream=s):
            binding.mhc_post_fwd(x, y, post, res, out)
            binding.mhc_post_bwd(g, x, y, post, res, gx, gy, gp, gr)
    for t in (out, gx, gy, gp, gr):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    e = [binding.post(x, y, post, res)] + list(binding.post_backward(g, x, y, post, res))
    for a, b in zip((out, gx, gy, gp, gr), e):
        assert sha(a) == sha(b)


# --------------------------------------------------------------------------
# post = sigmoid(alpha * mix + b) computed in the kernels
# --------------------------------------------------------------------------

from invariant_mhc_aggregate_gb300.autograd import mhc_post_sigmoid  # noqa: E402
from invariant_mhc_aggregate_gb300.inputs import coeff_inputs  # noqa: E402


def _scalar_buf(v: torch.Tensor) -> DevBuf:
    return DevBuf.of(v.reshape(-1).to(torch.float32))


def _np_ab(alpha, b):
    return np.float32(alpha.reshape(-1)[0].item()), f32(b)


def run_post_sigmoid_fwd(x, y, mix, alpha, b, res, offsets=(0, 0, 0)):
    """offsets: x, y, out."""
    T, n, H = x.shape
    bx, by, bo = DevBuf.of(x, offsets[0]), DevBuf.of(y, offsets[1]), DevBuf(T * n * H * 2, offsets[2])
    bm, ba, bb, br = DevBuf.of(mix), _scalar_buf(alpha), _scalar_buf(b), DevBuf.of(res)
    st = binding.post_sigmoid_fwd_raw(bx.ptr, by.ptr, bm.ptr, ba.ptr, bb.ptr, br.ptr, bo.ptr, T, n, H,
                                      DTYPE_CODE[x.dtype], stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    assert bo.guards_ok(), "forward wrote outside out"
    return bo.get(np.uint16, (T, n, H))


def run_post_sigmoid_bwd(g, x, y, mix, alpha, b, res, offsets=(0, 0, 0, 0, 0)):
    """offsets: g, x, y, grad_x, grad_y."""
    T, n, H = x.shape
    bg, bx, by = DevBuf.of(g, offsets[0]), DevBuf.of(x, offsets[1]), DevBuf.of(y, offsets[2])
    bm, ba, bb, br = DevBuf.of(mix), _scalar_buf(alpha), _scalar_buf(b), DevBuf.of(res)
    outs = [DevBuf(T * n * H * 2, offsets[3]), DevBuf(T * H * 2, offsets[4]), DevBuf(T * n * 4),
            DevBuf(T * n * 4), DevBuf(T * n * n * 4)]
    st = binding.post_sigmoid_bwd_raw(bg.ptr, bx.ptr, by.ptr, bm.ptr, ba.ptr, bb.ptr, br.ptr,
                                      *(o.ptr for o in outs), T, n, H, DTYPE_CODE[x.dtype], stream_handle())
    assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    assert all(o.guards_ok() for o in outs), "backward wrote outside its outputs"
    return (outs[0].get(np.uint16, (T, n, H)), outs[1].get(np.uint16, (T, H)), outs[2].get(np.float32, (T, n)),
            outs[3].get(np.float32, (T, n)), outs[4].get(np.float32, (T, n, n)))


SIG_CASES = [
    (5, 4096, (0, 0, 0)),      # 16-byte path
    (3, 7168, (0, 0, 0)),      # a forward block spans two tokens
    (9, 320, (0, 0, 0)),       # 40 vectors a row: forward warps straddle tokens, ragged last warp
    (4, 4104, (0, 0, 0)),      # 513 vectors a row
    (37, 64, (0, 0, 0)),       # 8 vectors a row: a forward block spans 33 tokens
    (6, 8, (0, 0, 0)),         # one vector a row
    (3, 4100, (0, 0, 0)),      # 2-byte path
    (2, 1279, (0, 2, 6)),
]


@pytest.mark.parametrize("recipe", ("normal", "wide"))
@pytest.mark.parametrize("dtype", DTYPES, ids=_ids)
@pytest.mark.parametrize("n", NS)
@pytest.mark.parametrize("T,H,offsets", SIG_CASES)
def test_post_sigmoid_all_paths(T, H, offsets, n, dtype, recipe):
    x, y, _, res, g = post_inputs(T, H, n, "normal", 1000 + T + H, dtype=dtype, with_grad=True)
    mix, alpha, b = coeff_inputs(T, n, recipe, 1001 + T)
    a_np, b_np = _np_ab(alpha, b)
    name = DTYPE_NAME[dtype]
    got = run_post_sigmoid_fwd(x, y, mix, alpha, b, res, offsets)
    want = oracle.post_sigmoid_fwd(u16(x), u16(y), f32(mix), a_np, b_np, f32(res), name)
    assert_bytes_equal(got, want, "out")
    got = run_post_sigmoid_bwd(g, x, y, mix, alpha, b, res, (0,) + tuple(offsets[:2]) + (offsets[2], 0))
    want = oracle.post_sigmoid_bwd(u16(g), u16(x), u16(y), f32(mix), a_np, b_np, f32(res), name)
    for a, w, what in zip(got, want, ("grad_x", "grad_y", "grad_z", "grad_mix", "grad_res")):
        assert_bytes_equal(a, w, what)


def test_post_sigmoid_full_size_against_oracle():
    T, H, n = 4096, 7168, 4
    x, y, _, res, g = post_inputs(T, H, n, "normal", 6, with_grad=True)
    mix, alpha, b = coeff_inputs(T, n, "normal", 7)
    xd, yd, rd, gd, md, ad, bd = (t.cuda() for t in (x, y, res, g, mix, alpha, b))
    out = binding.post_sigmoid(xd, yd, md, ad, bd, rd)
    grads = binding.post_sigmoid_backward(gd, xd, yd, md, ad, bd, rd)
    gb, ga = binding.sigmoid_param_grad(grads[2], md)
    torch.cuda.synchronize()
    a_np, b_np = _np_ab(alpha, b)
    o = oracle.default()
    assert_bytes_equal(u16(out), o.post_sigmoid_fwd(u16(x), u16(y), f32(mix), a_np, b_np, f32(res)), "out")
    want = o.post_sigmoid_bwd(u16(g), u16(x), u16(y), f32(mix), a_np, b_np, f32(res))
    for a, w, what in zip((u16(grads[0]), u16(grads[1]), f32(grads[2]), f32(grads[3]), f32(grads[4])), want,
                          ("grad_x", "grad_y", "grad_z", "grad_mix", "grad_res")):
        assert_bytes_equal(a, w, what)
    wgb, wga = o.sigmoid_param_grad(want[2], f32(mix))
    assert_bytes_equal(f32(gb), wgb, "grad_b")
    assert f32(ga).view(np.uint32)[0] == np.float32(wga).view(np.uint32)


@pytest.mark.parametrize("n", (1, 4, 8))
def test_post_sigmoid_batch_split_invariance(n):
    T, H = 64, 4096
    x, y, _, res, g = post_inputs(T, H, n, "normal", 1100 + n, with_grad=True)
    mix, alpha, b = coeff_inputs(T, n, "wide", 1101 + n)
    xd, yd, rd, gd, md, ad, bd = (t.cuda() for t in (x, y, res, g, mix, alpha, b))
    full = binding.post_sigmoid(xd, yd, md, ad, bd, rd)
    fgrads = binding.post_sigmoid_backward(gd, xd, yd, md, ad, bd, rd)
    for chunk in (1, 7, 64):
        for t0 in range(0, T, chunk):
            sl = slice(t0, min(T, t0 + chunk))
            xs, ys, ms, rs, gs = (t[sl].contiguous() for t in (xd, yd, md, rd, gd))
            assert sha(binding.post_sigmoid(xs, ys, ms, ad, bd, rs)) == sha(full[sl]), (chunk, t0)
            for p, f in zip(binding.post_sigmoid_backward(gs, xs, ys, ms, ad, bd, rs), fgrads):
                assert sha(p) == sha(f[sl]), (chunk, t0)


def test_post_sigmoid_autograd_matches_oracle():
    T, H, n = 2 * 11, 2048, 4
    x, y, _, res, g = post_inputs(T, H, n, "normal", 1200, with_grad=True)
    mix, alpha, b = coeff_inputs(T, n, "normal", 1201)
    xd = x.cuda().reshape(2, 11, n, H).requires_grad_(True)
    yd = y.cuda().reshape(2, 11, H).requires_grad_(True)
    md = mix.cuda().reshape(2, 11, n).requires_grad_(True)
    ad = alpha.reshape(()).cuda().requires_grad_(True)
    bd = b.cuda().requires_grad_(True)
    rd = res.cuda().reshape(2, 11, n, n).requires_grad_(True)
    out = mhc_post_sigmoid(xd, yd, md, ad, bd, rd)
    out.backward(g.cuda().reshape(2, 11, n, H))
    a_np, b_np = _np_ab(alpha, b)
    o = oracle.default()
    assert_bytes_equal(u16(out.detach().reshape(T, n, H)),
                       o.post_sigmoid_fwd(u16(x), u16(y), f32(mix), a_np, b_np, f32(res)), "out")
    wgx, wgy, wgz, wgm, wgr = o.post_sigmoid_bwd(u16(g), u16(x), u16(y), f32(mix), a_np, b_np, f32(res))
    wgb, wga = o.sigmoid_param_grad(wgz, f32(mix))
    assert_bytes_equal(u16(xd.grad.reshape(T, n, H)), wgx, "x.grad")
    assert_bytes_equal(u16(yd.grad.reshape(T, H)), wgy, "y.grad")
    assert_bytes_equal(f32(md.grad.reshape(T, n)), wgm, "mix.grad")
    assert_bytes_equal(f32(rd.grad.reshape(T, n, n)), wgr, "res.grad")
    assert_bytes_equal(f32(bd.grad), wgb, "b.grad")
    assert ad.grad.shape == () and f32(ad.grad).view(np.uint32) == np.float32(wga).view(np.uint32)


# --------------------------------------------------------------------------
# fuzzing and concurrency
# --------------------------------------------------------------------------

def test_post_fuzz_shapes_alignments_sources():
    rng = np.random.default_rng(2027)
    for case in range(40):
        n = int(rng.choice([1, 2, 4, 8]))
        dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float16
        H = int(rng.choice([int(rng.integers(1, 300)), 8 * int(rng.integers(1, 1100))]))
        T = int(rng.integers(1, 24))
        sig = bool(rng.random() < 0.4)
        x, y, post, res, g = post_inputs(T, H, n, str(rng.choice(["normal", "ragged"])),
                                         int(rng.integers(0, 10 ** 6)), dtype=dtype, with_grad=True)
        name = DTYPE_NAME[dtype]
        what = f"case {case}: n={n} {name} T={T} H={H} sigmoid={sig}"
        if sig:
            mix, alpha, b = coeff_inputs(T, n, str(rng.choice(["normal", "wide"])), int(rng.integers(0, 10 ** 6)))
            a_np, b_np = _np_ab(alpha, b)
            fo = tuple(int(rng.choice([0, 2, 8, 16])) for _ in range(3))
            got = run_post_sigmoid_fwd(x, y, mix, alpha, b, res, fo)
            assert_bytes_equal(got, oracle.post_sigmoid_fwd(u16(x), u16(y), f32(mix), a_np, b_np, f32(res), name),
                               "out " + what)
            bo = tuple(int(rng.choice([0, 2, 8, 16])) for _ in range(5))
            got = run_post_sigmoid_bwd(g, x, y, mix, alpha, b, res, bo)
            want = oracle.post_sigmoid_bwd(u16(g), u16(x), u16(y), f32(mix), a_np, b_np, f32(res), name)
            names = ("grad_x", "grad_y", "grad_z", "grad_mix", "grad_res")
        else:
            fo = tuple(int(rng.choice([0, 2, 8, 16])) if i in (0, 1, 4) else int(rng.choice([0, 4, 8]))
                       for i in range(5))
            got = run_post_fwd(x, y, post, res, fo)
            assert_bytes_equal(got, oracle.post_fwd(u16(x), u16(y), f32(post), f32(res), name), "out " + what)
            bo = tuple(int(rng.choice([0, 2, 8, 16])) if i in (0, 1, 2, 5, 6) else int(rng.choice([0, 4, 8]))
                       for i in range(9))
            got = run_post_bwd(g, x, y, post, res, bo)
            want = oracle.post_bwd(u16(g), u16(x), u16(y), f32(post), f32(res), name)
            names = ("grad_x", "grad_y", "grad_post", "grad_res")
        for a, w, nm in zip(got, want, names):
            assert_bytes_equal(a, w, f"{nm} {what}")


def test_post_concurrent_host_threads_on_separate_streams():
    import threading
    jobs = []
    for i in range(6):
        n = (4, 2, 8)[i % 3]
        x, y, post, res, g = (t.cuda() for t in post_inputs(96, 4096, n, "normal", 300 + i, with_grad=True))
        mix, alpha, b = (t.cuda() for t in coeff_inputs(96, n, "normal", 400 + i))
        jobs.append((x, y, post, res, g, mix, alpha, b, i % 2 == 1))
    torch.cuda.synchronize()

    def run(job, stream=None):
        x, y, post, res, g, mix, alpha, b, sig = job
        if sig:
            outs = [binding.post_sigmoid(x, y, mix, alpha, b, res, stream)]
            outs += list(binding.post_sigmoid_backward(g, x, y, mix, alpha, b, res, stream))
        else:
            outs = [binding.post(x, y, post, res, stream)] + list(binding.post_backward(g, x, y, post, res, stream))
        return outs

    refs = []
    for job in jobs:
        outs = run(job)
        torch.cuda.synchronize()
        refs.append([sha(o) for o in outs])
    results = [None] * len(jobs)
    errors = []

    def worker(i):
        try:
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(10):
                    outs = run(jobs[i], s)
            s.synchronize()
            results[i] = [sha(o) for o in outs]
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert results == refs
    assert binding.wait_timeouts() == 0


def test_post_split_launch_beyond_2e31_vectors():
    """The post forward indexes vectors with 32 bits and splits calls of 2^31
    vectors or more into launches over consecutive token ranges.  With n = 1,
    H = 16384 and the 16-byte path, T = 2^20 tokens make exactly 2^31 vectors:
    the second launch holds the last token (34 GB each for x, y and out).
    Checked for post given and for post computed from the mix."""
    T, H, n = 1 << 20, 16384, 1
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(321)
    x = torch.empty((T, n, H), dtype=torch.bfloat16, device=dev)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    step = 1 << 28
    for flat in (x.view(-1), y.view(-1)):
        for i in range(0, flat.numel(), step):
            m = min(step, flat.numel() - i)
            flat[i:i + m] = torch.randn(m, generator=gen, device=dev).to(torch.bfloat16)
    post = 2 * torch.rand((T, n), generator=gen, device=dev)
    res = torch.rand((T, n, n), generator=gen, device=dev)
    out = torch.empty_like(x)
    assert binding.post_fwd_path_raw(x.data_ptr(), y.data_ptr(), post.data_ptr(), res.data_ptr(),
                                     out.data_ptr(), T, n, H) == binding.MHC_PATH_VEC16
    V = H // 8
    boundary = (2 ** 31 - 1) // V          # first token of the second launch
    samples = (0, 1, boundary - 1, boundary, T - 1)
    binding.mhc_post_fwd(x, y, post, res, out)
    torch.cuda.synchronize()
    for t in samples:
        sl = slice(t, t + 1)
        want = oracle.post_fwd(u16(x[sl]), u16(y[sl]), f32(post[sl]), f32(res[sl]))
        assert_bytes_equal(u16(out[sl]), want, f"token {t}")
    mix = torch.randn((T, n), generator=gen, device=dev) * 3
    alpha = torch.full((1,), 1.25, device=dev)
    b = torch.full((1,), -0.5, device=dev)
    binding.mhc_post_sigmoid_fwd(x, y, mix, alpha, b, res, out)
    torch.cuda.synchronize()
    for t in samples:
        sl = slice(t, t + 1)
        want = oracle.post_sigmoid_fwd(u16(x[sl]), u16(y[sl]), f32(mix[sl]), np.float32(1.25),
                                       np.float32([-0.5]), f32(res[sl]))
        assert_bytes_equal(u16(out[sl]), want, f"sigmoid post, token {t}")
    del x, y, out, post, res, mix
    torch.cuda.empty_cache()


# --- magnitudes around the exact-product check of the fused first level

# (row kind, row index, scale): whole rows scaled by a power of two; FP16
# cases stay finite (subnormals and underflow to zero, values up to ~2^15)
MAGNITUDE_CASES = {
    torch.bfloat16: (("x", 3, 2.0 ** -40), ("x", 5, 2.0 ** -62), ("y", 0, 2.0 ** -66),
                     ("g", 2, 2.0 ** -75), ("x", 1, 2.0 ** -130), ("g", 6, 2.0 ** 62),
                     ("x", 0, 2.0 ** 66), ("y", 0, 2.0 ** 100)),
    torch.float16: (("x", 3, 2.0 ** -8), ("x", 5, 2.0 ** -14), ("y", 0, 2.0 ** -20),
                    ("g", 2, 2.0 ** -30), ("x", 1, 2.0 ** 4), ("g", 6, 2.0 ** 8),
                    ("x", 0, 2.0 ** 12), ("y", 0, 2.0 ** 13)),
}


@pytest.mark.parametrize("n", (4, 8))
@pytest.mark.parametrize("dtype", DTYPES, ids=_ids)
def test_post_bwd_magnitude_classes(n, dtype):
    """Blocks of tokens whose g, x or y rows are scaled far from 1 (BF16: into
    the subnormal range, around the 2^-63 and 2^64 bounds of the check that
    lets a chunk take the fused first level, and beyond), plus exact zeros and
    lone extreme values in one position half: every output against the
    oracle.  The n = 8 kernel takes the fused or the unfused level chunk by
    chunk; both must give the oracle's bytes."""
    cases = MAGNITUDE_CASES[dtype]
    T, H = 8 * len(cases), 2048
    x, y, post, res, g = post_inputs(T, H, n, "normal", 21, dtype=dtype, with_grad=True)
    x, y, g = x.float(), y.float(), g.float()
    rows = {"x": x, "y": y, "g": g}
    for b, (kind, r, scale) in enumerate(cases):
        sl = slice(8 * b, 8 * b + 8)
        if kind == "y":
            rows[kind][sl] *= scale
        else:
            rows[kind][sl, r % n] *= scale
    # exact zeros, and lone extremes at single positions of otherwise normal rows
    x[0, 0, ::5] = 0.0
    g[1, n - 1, 7] = 2.0 ** -100 if dtype == torch.bfloat16 else 2.0 ** -24
    x[2, 0, 1029] = 2.0 ** 70 if dtype == torch.bfloat16 else 60000.0
    y[3, 4] = -(2.0 ** -64) if dtype == torch.bfloat16 else 2.0 ** -20
    x, y, g = (t.to(dtype) for t in (x, y, g))
    got = run_post_bwd(g, x, y, post, res)
    want = oracle.default().post_bwd(u16(g), u16(x), u16(y), f32(post), f32(res), DTYPE_NAME[dtype])
    for a, w, what in zip(got, want, ("grad_x", "grad_y", "grad_post", "grad_res")):
        assert_bytes_equal(a, w, f"{what} n={n}")

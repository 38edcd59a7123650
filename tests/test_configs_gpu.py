"""The five benchmark workloads, each checked in full on the GPU through the C ABI:

* every output of every shape byte-identical to the CPU oracle (no sampling:
  the oracle runs over contiguous token blocks on all host threads, which is
  exact because every output of a token depends on that token alone);
* 100 repeat calls on the same buffers give the same bytes;
* the full batch, one-token calls, 64-token calls and 4096-token calls give
  the same bytes (the calls see other alignments, grids and launch shapes).

Source of the contract: "Add batch-invariant h_aggregate kernel" --
Correctness (run-to-run and batch-split byte equality), Summary (shapes,
formula) and the Performance table's (T, H) sweep; the backward's checks are
the reviewer's request on the same page.
"""

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
from _gpu import assert_bytes_equal, lib, stream_handle, u16, f32
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.inputs import (backward_inputs, forward_inputs,
                                                  post_inputs, workload)

pytestmark = pytest.mark.gpu

SPLITS = (1, 64, 4096)
REPEATS = 100


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


def by_token_blocks(fn, *arrays):
    """Run a per-token oracle function over contiguous token blocks on host
    threads (the oracle's C calls release the GIL) and join the outputs."""
    T = arrays[0].shape[0]
    threads = max(1, min(os.cpu_count() or 1, 64))
    step = max(1, -(-T // (4 * threads)))
    ranges = [(t0, min(T, t0 + step)) for t0 in range(0, T, step)]
    with ThreadPoolExecutor(threads) as ex:
        parts = list(ex.map(lambda r: fn(*(a[r[0]:r[1]] for a in arrays)), ranges))
    if isinstance(parts[0], tuple):
        return tuple(np.concatenate([p[i] for p in parts]) for i in range(len(parts[0])))
    return np.concatenate(parts)


def same_bytes(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.contiguous().view(torch.uint8), b.contiguous().view(torch.uint8))


# --- forward: configs 1-4

def fwd_split(r_d, p_d, chunk):
    """The forward as calls of `chunk` tokens each, through the raw C ABI."""
    T, _, H = r_d.shape
    out = torch.full((T, H), -1, dtype=torch.int16, device=r_d.device).view(torch.bfloat16)
    rp, pp, op = r_d.data_ptr(), p_d.data_ptr(), out.data_ptr()
    s = stream_handle()
    for t0 in range(0, T, chunk):
        c = min(chunk, T - t0)
        st = binding.fwd_raw(rp + t0 * 4 * H * 2, pp + t0 * 16, op + t0 * H * 2, c, H, s)
        assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    return out


def check_fwd_config(res, pre, what):
    r_d, p_d = res.cuda(), pre.cuda()
    T, _, H = res.shape
    full = binding.h_aggregate(r_d, p_d)
    torch.cuda.synchronize()
    assert_bytes_equal(u16(full), by_token_blocks(oracle.fwd, u16(res), f32(pre)),
                       f"{what}: vs oracle")
    out = torch.empty_like(full)
    for i in range(REPEATS):
        out.view(torch.int16).fill_(-1 - i)
        binding.mhc_h_aggregate_fwd(r_d, p_d, out)
        assert same_bytes(out, full), f"{what}: repeat call {i} differs"
    for chunk in SPLITS:
        if chunk < T or chunk == 1:
            assert same_bytes(fwd_split(r_d, p_d, chunk), full), \
                f"{what}: {chunk}-token calls differ from the full batch"


def test_config1_t129_h4096():
    w = workload("fwd_t129_h4096")
    (T, H), = w.shapes
    check_fwd_config(*forward_inputs(T, H, w.recipe, w.seed), f"T={T} H={H}")


@pytest.mark.parametrize("T,H", workload("fwd_ragged").shapes)
def test_config2_ragged(T, H):
    w = workload("fwd_ragged")
    check_fwd_config(*forward_inputs(T, H, w.recipe, w.seed), f"ragged T={T} H={H}")


@pytest.mark.parametrize("T,H", workload("fwd_decode").shapes)
def test_config3_decode(T, H):
    w = workload("fwd_decode")
    check_fwd_config(*forward_inputs(T, H, w.recipe, w.seed), f"decode T={T} H={H}")


@pytest.mark.parametrize("T", [1024, 4096, 16384])
def test_config4_prefill(T):
    w = workload("fwd_prefill")
    check_fwd_config(*forward_inputs(T, 7168, w.recipe, w.seed), f"prefill T={T}")


def test_config4_prefill_t65536():
    """The largest workload (3.76 GB residual), drawn on the device as the
    benchmark draws it, compared with the oracle on every token."""
    w = workload("fwd_prefill")
    T, H = 65536, 7168
    res_d, pre_d = forward_inputs(T, H, w.recipe, w.seed, device="cuda")
    check_fwd_config(res_d, pre_d, f"prefill T={T}")
    del res_d, pre_d
    torch.cuda.empty_cache()


# --- backward: config 5

def bwd_split(g_d, r_d, p_d, chunk):
    T, _, H = r_d.shape
    gr = torch.full((T, 4, H), -1, dtype=torch.int16, device=r_d.device).view(torch.bfloat16)
    gp = torch.full((T, 4), float("nan"), dtype=torch.float32, device=r_d.device)
    gptr, rptr, pptr = g_d.data_ptr(), r_d.data_ptr(), p_d.data_ptr()
    s = stream_handle()
    for t0 in range(0, T, chunk):
        c = min(chunk, T - t0)
        st = binding.bwd_raw(gptr + t0 * H * 2, rptr + t0 * 4 * H * 2, pptr + t0 * 16,
                             gr.data_ptr() + t0 * 4 * H * 2, gp.data_ptr() + t0 * 16, c, H, s)
        assert st == binding.MHC_OK, st
    torch.cuda.synchronize()
    return gr, gp


def test_config5_backward_t4096_h7168():
    w = workload("bwd_t4096_h7168")
    (T, H), = w.shapes
    g, res, pre = backward_inputs(T, H, w.recipe, w.seed)
    g_d, r_d, p_d = g.cuda(), res.cuda(), pre.cuda()
    gr, gp = binding.h_aggregate_backward(g_d, r_d, p_d)
    torch.cuda.synchronize()
    want_gr, want_gp = by_token_blocks(oracle.bwd, u16(g), u16(res), f32(pre))
    assert_bytes_equal(u16(gr), want_gr, "grad_residual vs oracle")
    assert_bytes_equal(f32(gp), want_gp, "grad_pre vs oracle (ORDER-256)")
    gr2, gp2 = torch.empty_like(gr), torch.empty_like(gp)
    for i in range(REPEATS):
        gr2.view(torch.int16).fill_(-1 - i)
        gp2.fill_(float(i))
        binding.mhc_h_aggregate_bwd(g_d, r_d, p_d, gr2, gp2)
        assert same_bytes(gr2, gr) and same_bytes(gp2, gp), f"repeat call {i} differs"
    for chunk in SPLITS:
        sgr, sgp = bwd_split(g_d, r_d, p_d, chunk)
        assert same_bytes(sgr, gr), f"grad_residual differs with {chunk}-token calls"
        assert same_bytes(sgp, gp), f"grad_pre differs with {chunk}-token calls"


# --- the mHC post at n = 8, the benchmark's n = 8 shape, every token

def test_post_n8_t4096_h7168_every_token():
    T, H, n = 4096, 7168, 8
    x, y, post, res, g = post_inputs(T, H, n, "normal", 6, with_grad=True)
    xd, yd, pd, rd, gd = (t.cuda() for t in (x, y, post, res, g))
    out = binding.post(xd, yd, pd, rd)
    gx, gy, gp, gr = binding.post_backward(gd, xd, yd, pd, rd)
    torch.cuda.synchronize()
    o = oracle.default()
    want = by_token_blocks(o.post_fwd, u16(x), u16(y), f32(post), f32(res))
    assert_bytes_equal(u16(out), want, "out")
    want = by_token_blocks(o.post_bwd, u16(g), u16(x), u16(y), f32(post), f32(res))
    got = (u16(gx), u16(gy), f32(gp), f32(gr))
    for a, b, what in zip(got, want, ("grad_x", "grad_y", "grad_post", "grad_res")):
        assert_bytes_equal(a, b, what)
    # repeat calls and 64-token splits give the same bytes
    for i in range(10):
        gx2, gy2, gp2, gr2 = binding.post_backward(gd, xd, yd, pd, rd)
        out2 = binding.post(xd, yd, pd, rd)
        assert all(same_bytes(a, b) for a, b in
                   ((gx2, gx), (gy2, gy), (gp2, gp), (gr2, gr), (out2, out))), i
    for t0 in range(0, T, 64):
        sl = slice(t0, t0 + 64)
        o2 = binding.post(xd[sl], yd[sl], pd[sl], rd[sl])
        b2 = binding.post_backward(gd[sl], xd[sl], yd[sl], pd[sl], rd[sl])
        assert same_bytes(o2, out[sl]), t0
        assert all(same_bytes(a, b[sl]) for a, b in zip(b2, (gx, gy, gp, gr))), t0

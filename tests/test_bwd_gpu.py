"""Backward parity on the GPU: grad_residual and grad_pre from the sm_103a
kernels against the CPU oracle, byte for byte, through the C ABI
(gradient_accuracy and gradient_invariance).

Source: "Add batch-invariant h_aggregate kernel" -- the reviewer's request for
a backward with gradient accuracy and invariance checks; the formula is the
derivative of the page's Summary formula, grad_pre summed in ORDER-256.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import _pins
from _gpu import assert_bytes_equal, lib, run_bwd, sha, u16, f32
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.inputs import backward_inputs, workload

pytestmark = pytest.mark.gpu

VEC32, VEC16, ELEMENT = binding.MHC_PATH_VEC32, binding.MHC_PATH_VEC16, binding.MHC_PATH_ELEMENT


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


def oracle_bwd(g, res, pre):
    return oracle.bwd(u16(g), u16(res), f32(pre))


def grad_pre_fp64_check(gp: np.ndarray, g: torch.Tensor, res: torch.Tensor):
    """|got - exact| <= 1e-3 * max(|exact|, sum_h |g r|), exact = FP64 sum of the
    exact products.  Also returns the plain max relative error and how many
    entries exceed 1e-3 plainly (sums that cancel to near zero)."""
    gw = f32(g.float()).astype(np.float64)
    rw = f32(res.float()).astype(np.float64)
    q = gw[:, None, :] * rw
    exact = q.sum(axis=2)
    mag = np.abs(q).sum(axis=2)
    err = np.abs(gp.astype(np.float64) - exact)
    assert np.all(err <= 1e-3 * np.maximum(np.abs(exact), mag))
    rel = err / np.maximum(np.abs(exact), np.finfo(np.float64).tiny)
    return float(rel.max()), int(np.sum(rel > 1e-3))


# --- workload bwd_t4096_h7168: T=4096, H=7168, seed 4

@pytest.fixture(scope="module")
def bwd_workload():
    w = workload("bwd_t4096_h7168")
    (T, H), = w.shapes
    return backward_inputs(T, H, w.recipe, w.seed)


def test_t4096_bit_exact(bwd_workload):
    g, res, pre = bwd_workload
    gd, rd, pd = g.cuda(), res.cuda(), pre.cuda()
    gr, gp = binding.h_aggregate_backward(gd, rd, pd)
    torch.cuda.synchronize()
    want_gr, want_gp = oracle_bwd(g, res, pre)
    assert_bytes_equal(u16(gr), want_gr, "grad_residual")
    assert_bytes_equal(f32(gp), want_gp, "grad_pre (ORDER-256)")
    grad_pre_fp64_check(f32(gp), g, res)


def test_t4096_split_invariance(bwd_workload):
    """1-, 64- and 4096-token calls give identical bytes."""
    g, res, pre = bwd_workload
    gd, rd, pd = g.cuda(), res.cuda(), pre.cuda()
    T, _, H = res.shape
    ref_gr, ref_gp = binding.h_aggregate_backward(gd, rd, pd)
    for chunk in (1, 64):
        gr = torch.empty_like(ref_gr)
        gp = torch.empty_like(ref_gp)
        for t0 in range(0, T, chunk):
            sl = slice(t0, t0 + chunk)
            binding.mhc_h_aggregate_bwd(gd[sl], rd[sl], pd[sl], gr[sl], gp[sl])
        torch.cuda.synchronize()
        assert sha(gr) == sha(ref_gr), f"grad_residual differs with {chunk}-token calls"
        assert sha(gp) == sha(ref_gp), f"grad_pre differs with {chunk}-token calls"


def test_repeat_100_calls_byte_identical():
    g, res, pre = backward_inputs(64, 7168, "normal", 14, device="cuda")
    gr = torch.empty((64, 4, 7168), dtype=torch.bfloat16, device="cuda")
    gp = torch.empty((64, 4), dtype=torch.float32, device="cuda")
    digests = set()
    for _ in range(100):
        gr.zero_()
        gp.zero_()
        binding.mhc_h_aggregate_bwd(g, res, pre, gr, gp)
        digests.add(sha(gr) + sha(gp))
    assert len(digests) == 1


# --- shapes and paths

@pytest.mark.parametrize("T,H", [(1, 1), (2, 7), (3, 8), (1, 13), (4, 16), (5, 255), (3, 1279),
                                 (1, 2048), (2, 2050), (2, 2064), (2, 3072), (3, 4096),
                                 (1, 4097), (2, 4104), (2, 4112), (9, 7168), (1, 16392),
                                 (2, 65536)])
def test_shapes_bit_exact(T, H):
    g, res, pre = backward_inputs(T, H, "ragged", 15)
    gr, gp = run_bwd(g, res, pre)
    want_gr, want_gp = oracle_bwd(g, res, pre)
    assert_bytes_equal(gr, want_gr, f"grad_residual T={T} H={H}")
    assert_bytes_equal(gp, want_gp, f"grad_pre T={T} H={H}")


@pytest.mark.parametrize("T,H", [(7, 2048), (3, 7168), (2, 4104), (2, 24), (1, 4112)])
def test_paths_agree(T, H):
    g, res, pre = backward_inputs(T, H, "decode", 16)
    want_gr, want_gp = oracle_bwd(g, res, pre)
    for offsets in ((0, 0, 0, 0, 0), (0, 0, 4, 0, 4), (16, 0, 0, 0, 0), (0, 16, 0, 16, 0),
                    (2, 0, 0, 0, 0), (0, 4, 0, 0, 0), (0, 0, 0, 8, 0)):
        gr, gp = run_bwd(g, res, pre, offsets=offsets)
        assert_bytes_equal(gr, want_gr, f"grad_residual offsets={offsets}")
        assert_bytes_equal(gp, want_gp, f"grad_pre offsets={offsets}")


def test_order_cases_on_gpu():
    """The hand-worked ORDER-256 cases (tests/golden) through both kernel paths."""
    for name, H, k, carrier, positions, expected in _pins.golden_rows("grad_pre_order_cases.txt"):
        H, k = int(H), int(k)
        vals = np.zeros(H, dtype=np.uint16)
        for item in positions.split(","):
            pos, v = item.split(":")
            if pos == "*":
                vals[:] = int(v, 16)
            else:
                vals[int(pos)] = int(v, 16)
        g = np.full((1, H), 0x3F80, dtype=np.uint16)
        res = np.zeros((1, 4, H), dtype=np.uint16)
        if carrier == "r":
            res[0, k] = vals
        else:
            g[0] = vals
            res[0, k] = 0x3F80
        pre = np.ones((1, 4), dtype=np.float32)
        gt = torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16)
        rt = torch.from_numpy(res.view(np.int16).copy()).view(torch.bfloat16)
        want = np.zeros(4, dtype=np.uint32)
        want[k] = int(expected, 16)
        offsets_list = [(2, 0, 0, 0, 0)]
        if H % 8 == 0:
            offsets_list += [(0, 0, 0, 0, 0), (16, 16, 0, 16, 0)]
        for offsets in offsets_list:
            _, gp = run_bwd(gt, rt, torch.from_numpy(pre), offsets=offsets)
            assert np.array_equal(gp.view(np.uint32)[0], want), (name, offsets)


def test_grad_residual_worked_examples_on_gpu():
    rows = list(_pins.golden_rows("grad_residual_worked_examples.txt"))
    T, H = len(rows), 16
    rng = np.random.default_rng(41)
    g = _pins.random_bf16(rng, (T, H))
    res = _pins.random_bf16(rng, (T, 4, H))
    pre = rng.random((T, 4), dtype=np.float32)
    for t, (name, pbits, gbits, ebits) in enumerate(rows):
        pre[t, 1] = _pins.f32_from_bits(int(pbits, 16))
        g[t, 5] = int(gbits, 16)
    gt = torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16)
    rt = torch.from_numpy(res.view(np.int16).copy()).view(torch.bfloat16)
    for offsets in ((0, 0, 0, 0, 0), (16, 16, 0, 16, 0), (2, 0, 0, 2, 0)):
        gr, gp = run_bwd(gt, rt, torch.from_numpy(pre), offsets=offsets)
        for t, (name, pbits, gbits, ebits) in enumerate(rows):
            assert int(gr[t, 1, 5]) == int(ebits, 16), (name, offsets)
        want_gr, want_gp = oracle.bwd(g, res, pre)
        assert_bytes_equal(gr, want_gr, "grad_residual worked batch")
        assert_bytes_equal(gp, want_gp, "grad_pre worked batch")


def test_integer_valued_grad_pre_exact():
    """Integer g and r in [-8, 8]: the FP32 sums are exact, whatever the order."""
    rng = np.random.default_rng(42)
    T, H = 6, 7168
    gi = rng.integers(-8, 9, size=(T, H))
    ri = rng.integers(-8, 9, size=(T, 4, H))
    lut = np.array([_pins.bf16_bits_of(float(v)) for v in range(-8, 9)], dtype=np.uint16)
    g, res = lut[gi + 8], lut[ri + 8]
    pre = rng.random((T, 4), dtype=np.float32)
    gt = torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16)
    rt = torch.from_numpy(res.view(np.int16).copy()).view(torch.bfloat16)
    _, gp = run_bwd(gt, rt, torch.from_numpy(pre))
    assert np.array_equal(gp.astype(np.float64), np.einsum("th,tkh->tk", gi, ri).astype(np.float64))


def test_zero_tokens_launches_nothing():
    assert binding.bwd_raw(0, 0, 0, 0, 0, 0, 7168, 0) == binding.MHC_OK

"""The autograd wrapper on the GPU, the reviewer's four checks, and a training run.

"Add batch-invariant h_aggregate kernel", reviewer comment: add the backward
"so that training loss can converge", and check forward_accuracy,
forward_invariance, gradient_accuracy and gradient_invariance.  Accuracy here
is measured against exact FP64 arithmetic (products of BF16 and FP32 values are
exact in FP64); byte parity with the CPU oracle is checked as well.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import _pins
from _gpu import assert_bytes_equal, lib, u16, f32
from invariant_mhc_aggregate_gb300.autograd import h_aggregate
from invariant_mhc_aggregate_gb300.inputs import backward_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


def _run(g, res, pre):
    r = res.cuda().requires_grad_(True)
    p = pre.cuda().requires_grad_(True)
    out = h_aggregate(r, p)
    out.backward(g.cuda())
    torch.cuda.synchronize()
    return out.detach(), r.grad, p.grad


def test_autograd_matches_oracle_bytes():
    g, res, pre = backward_inputs(37, 7168, "normal", 31)
    out, gr, gp = _run(g, res, pre)
    assert out.dtype == torch.bfloat16 and gr.dtype == torch.bfloat16 and gp.dtype == torch.float32
    assert_bytes_equal(u16(out), oracle.fwd(u16(res), f32(pre)), "autograd forward")
    want_gr, want_gp = oracle.bwd(u16(g), u16(res), f32(pre))
    assert_bytes_equal(u16(gr), want_gr, "autograd grad_residual")
    assert_bytes_equal(f32(gp), want_gp, "autograd grad_pre")


def test_leading_batch_dims_and_partial_grads():
    g, res, pre = backward_inputs(6, 1024, "decode", 32)
    r = res.cuda().reshape(2, 3, 4, 1024)
    p = pre.cuda().reshape(2, 3, 4).requires_grad_(True)
    out = h_aggregate(r, p)
    assert out.shape == (2, 3, 1024)
    out.backward(g.cuda().reshape(2, 3, 1024))
    _, want_gp = oracle.bwd(u16(g), u16(res), f32(pre))
    assert np.array_equal(f32(p.grad.reshape(6, 4)).view(np.uint32), want_gp.view(np.uint32))


def four_way_report(T=256, H=7168, seed=33):
    """forward/gradient accuracy against exact FP64 and forward/gradient
    invariance under repeats and batch splits."""
    g, res, pre = backward_inputs(T, H, "normal", seed)
    out, gr, gp = _run(g, res, pre)
    rw = _pins.bf16_widen(u16(res)).astype(np.float64)
    gw = _pins.bf16_widen(u16(g)).astype(np.float64)
    pw = f32(pre).astype(np.float64)
    U = 2.0 ** -24
    # forward accuracy: |out - exact| against 1/2 BF16 ulp + the FP32 tree's bound
    prod = pw[:, :, None] * rw
    exact = prod.sum(axis=1)
    o64 = _pins.bf16_widen(u16(out)).astype(np.float64)
    fbound = 0.5 * _pins.bf16_ulp(o64) + 3.01 * U * np.abs(prod).sum(axis=1)
    fwd_ratio = float(np.max(np.abs(o64 - exact) / fbound))
    # gradient accuracy: grad_residual within one BF16 ulp of the exact product,
    # grad_pre within 1e-3 of the FP64 sum relative to max(|sum|, sum |g r|)
    gr64 = _pins.bf16_widen(u16(gr)).astype(np.float64)
    exact_gr = pw[:, :, None] * gw[:, None, :]
    gr_ratio = float(np.max(np.abs(gr64 - exact_gr) / _pins.bf16_ulp(gr64).clip(min=2.0 ** -133)))
    q = gw[:, None, :] * rw
    exact_gp = q.sum(axis=2)
    mag = np.abs(q).sum(axis=2)
    gp_err = np.abs(f32(gp).astype(np.float64) - exact_gp) / np.maximum(np.abs(exact_gp), mag)
    # invariance: repeats and one-token / 16-token splits are byte-identical
    fwd_inv = bwd_inv = True
    for _ in range(3):
        o2, gr2, gp2 = _run(g, res, pre)
        fwd_inv &= torch.equal(o2.view(torch.int16), out.view(torch.int16))
        bwd_inv &= torch.equal(gr2.view(torch.int16), gr.view(torch.int16)) and torch.equal(gp2, gp)
    for chunk in (1, 16):
        for t0 in range(0, T, chunk * 7):
            sl = slice(t0, t0 + chunk)
            o3, gr3, gp3 = _run(g[sl], res[sl], pre[sl])
            fwd_inv &= torch.equal(o3.view(torch.int16), out[sl].view(torch.int16))
            bwd_inv &= torch.equal(gr3.view(torch.int16), gr[sl].view(torch.int16))
            bwd_inv &= torch.equal(gp3.view(torch.int32), gp[sl].view(torch.int32))
    return {"forward_accuracy": {"max_err_over_bound": fwd_ratio},
            "forward_invariance": bool(fwd_inv),
            "gradient_accuracy": {"grad_residual_max_err_ulps": gr_ratio,
                                  "grad_pre_max_rel_err": float(gp_err.max())},
            "gradient_invariance": bool(bwd_inv)}


def test_four_way_report():
    rep = four_way_report()
    print(rep)
    assert rep["forward_accuracy"]["max_err_over_bound"] <= 1.0
    assert rep["forward_invariance"]
    assert rep["gradient_accuracy"]["grad_residual_max_err_ulps"] <= 1.0
    assert rep["gradient_accuracy"]["grad_pre_max_rel_err"] <= 1e-3
    assert rep["gradient_invariance"]


def test_training_loss_converges():
    """Fit pre by gradient descent through the op: the loss falls by orders of
    magnitude (the residual's BF16 gradient also flows)."""
    gen = torch.Generator(device="cuda").manual_seed(7)
    T, H = 64, 1024
    residual = torch.randn((T, 4, H), device="cuda", generator=gen).to(torch.bfloat16)
    pre_true = torch.rand((T, 4), device="cuda", generator=gen)
    target = h_aggregate(residual, pre_true).float()
    pre = torch.full((T, 4), 0.5, device="cuda", requires_grad=True)
    res_param = residual.clone().requires_grad_(True)
    opt = torch.optim.Adam([pre], lr=0.05)
    losses = []
    for _ in range(300):
        opt.zero_grad()
        loss = (h_aggregate(res_param, pre).float() - target).square().mean()
        loss.backward()
        opt.step()
        losses.append(float(loss.detach()))
    assert res_param.grad is not None and res_param.grad.dtype == torch.bfloat16
    assert math.isfinite(losses[-1])
    assert losses[-1] < 1e-3 * losses[0], (losses[0], losses[-1])

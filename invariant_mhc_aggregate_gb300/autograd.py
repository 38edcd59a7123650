"""PyTorch autograd wrapper over the C ABI, for training.

"Add batch-invariant h_aggregate kernel" (reviewer comment) asks for the
backward of h_aggregate "so that training loss can converge".  `h_aggregate`
below is differentiable in both inputs: the forward and the backward each run
as one kernel of ``libmhc_h_aggregate.so`` (through ``binding``); PyTorch only
allocates the outputs and tracks the graph.

    out = h_aggregate(residual, pre)      # residual [T,4,H] bf16, pre [T,4] fp32
    out.float().square().mean().backward()
    residual.grad  # bf16 [T,4,H] = bf16(fp32(pre * g))
    pre.grad       # fp32 [T,4]   = ORDER-256 sums of g * residual

Inputs may have any leading batch shape: ``residual [..., n, H]`` and
``pre [..., n]`` are flattened to tokens and the results reshaped back.  The
pages' op has n = 4 streams and BF16 storage; n in {1, 2, 8} and FP16 storage
run the library's general form (balanced pairwise tree, same roundings).
"""

from __future__ import annotations

import torch

from . import binding


class HAggregate(torch.autograd.Function):
    @staticmethod
    def forward(ctx, residual: torch.Tensor, pre: torch.Tensor) -> torch.Tensor:
        if residual.dtype not in (torch.bfloat16, torch.float16) or pre.dtype != torch.float32:
            raise TypeError("h_aggregate expects residual bf16/f16 [...,n,H] and pre fp32 [...,n]")
        if residual.dim() < 2 or residual.shape[:-1] != pre.shape:
            raise ValueError(f"shape mismatch: residual {tuple(residual.shape)}, pre {tuple(pre.shape)}")
        lead = residual.shape[:-2]
        n, H = residual.shape[-2], residual.shape[-1]
        r = residual.reshape(-1, n, H).contiguous()
        p = pre.reshape(-1, n).contiguous()
        out = binding.aggregate(r, p)
        ctx.save_for_backward(r, p)
        ctx.lead = lead
        return out.reshape(*lead, H)

    @staticmethod
    def backward(ctx, grad_out: torch.Tensor):
        r, p = ctx.saved_tensors
        n, H = r.shape[-2], r.shape[-1]
        if grad_out.dtype != r.dtype:
            raise TypeError(f"the output gradient must be {r.dtype}, got {grad_out.dtype}")
        g = grad_out.reshape(-1, H).contiguous()
        grad_residual, grad_pre = binding.aggregate_backward(g, r, p)
        gr = grad_residual.reshape(*ctx.lead, n, H) if ctx.needs_input_grad[0] else None
        gp = grad_pre.reshape(*ctx.lead, n) if ctx.needs_input_grad[1] else None
        return gr, gp


def h_aggregate(residual: torch.Tensor, pre: torch.Tensor) -> torch.Tensor:
    """Differentiable batch-invariant H Aggregate (see the module docstring)."""
    return HAggregate.apply(residual, pre)


class HAggregateSigmoid(torch.autograd.Function):
    """out = aggregate(residual, sigmoid(alpha * mix + b)), with the pre
    coefficients computed inside the kernels ("perf: fuse mHC coefficient
    backward epilogue", Summary: the pre sigmoid's derivative, grad_mix and the
    gradients of b and alpha).  The backward is one fused kernel for
    grad_residual, grad_z and grad_mix, and one kernel summing grad_b and
    grad_alpha over tokens in a fixed order."""

    @staticmethod
    def forward(ctx, residual, mix, alpha, b):
        if residual.dtype not in (torch.bfloat16, torch.float16) or mix.dtype != torch.float32:
            raise TypeError("expects residual bf16/f16 [...,n,H] and mix fp32 [...,n]")
        if residual.dim() < 2 or residual.shape[:-1] != mix.shape:
            raise ValueError(f"shape mismatch: residual {tuple(residual.shape)}, mix {tuple(mix.shape)}")
        lead = residual.shape[:-2]
        n, H = residual.shape[-2], residual.shape[-1]
        r = residual.reshape(-1, n, H).contiguous()
        m = mix.reshape(-1, n).contiguous()
        a = alpha.reshape(1).contiguous()
        bb = b.contiguous()
        out = binding.aggregate_sigmoid(r, m, a, bb)
        ctx.save_for_backward(r, m, a, bb)
        ctx.lead = lead
        ctx.alpha_shape = alpha.shape
        return out.reshape(*lead, H)

    @staticmethod
    def backward(ctx, grad_out):
        r, m, a, bb = ctx.saved_tensors
        n, H = r.shape[-2], r.shape[-1]
        if grad_out.dtype != r.dtype:
            raise TypeError(f"the output gradient must be {r.dtype}, got {grad_out.dtype}")
        g = grad_out.reshape(-1, H).contiguous()
        grad_residual, grad_z, grad_mix = binding.aggregate_sigmoid_backward(g, r, m, a, bb)
        grad_alpha = grad_b = None
        if ctx.needs_input_grad[2] or ctx.needs_input_grad[3]:
            grad_b, grad_alpha = binding.sigmoid_param_grad(grad_z, m)
            grad_alpha = grad_alpha.reshape(ctx.alpha_shape)
        gr = grad_residual.reshape(*ctx.lead, n, H) if ctx.needs_input_grad[0] else None
        gm = grad_mix.reshape(*ctx.lead, n) if ctx.needs_input_grad[1] else None
        return (gr, gm, grad_alpha if ctx.needs_input_grad[2] else None,
                grad_b if ctx.needs_input_grad[3] else None)


def h_aggregate_sigmoid(residual: torch.Tensor, mix: torch.Tensor, alpha: torch.Tensor,
                        b: torch.Tensor) -> torch.Tensor:
    """Differentiable aggregate with pre = sigmoid(alpha * mix + b) computed in the kernel."""
    return HAggregateSigmoid.apply(residual, mix, alpha, b)


class MhcPost(torch.autograd.Function):
    """out[..., k, :] = tree_n(res[..., k, j] * x[..., j, :]) + post[..., k] * y —
    the layer output y expanded back onto the n streams (the library's reading
    of the "MHC Post" stage named in "Add batch-invariant h_aggregate kernel",
    Summary).  Forward and backward are one kernel each; the backward gives
    all four gradients, grad_post and grad_res summed over H in ORDER-256."""

    @staticmethod
    def forward(ctx, x, y, post, res):
        if x.dtype not in (torch.bfloat16, torch.float16) or y.dtype != x.dtype:
            raise TypeError("expects x [...,n,H] and y [...,H] of one type, bf16 or f16")
        if post.dtype != torch.float32 or res.dtype != torch.float32:
            raise TypeError("expects post [...,n] and res [...,n,n] fp32")
        if x.dim() < 2:
            raise ValueError(f"x must be [...,n,H], got {tuple(x.shape)}")
        lead = x.shape[:-2]
        n, H = x.shape[-2], x.shape[-1]
        if y.shape != (*lead, H) or post.shape != (*lead, n) or res.shape != (*lead, n, n):
            raise ValueError(f"shape mismatch: x {tuple(x.shape)}, y {tuple(y.shape)}, "
                             f"post {tuple(post.shape)}, res {tuple(res.shape)}")
        xx = x.reshape(-1, n, H).contiguous()
        yy = y.reshape(-1, H).contiguous()
        pp = post.reshape(-1, n).contiguous()
        rr = res.reshape(-1, n, n).contiguous()
        out = binding.post(xx, yy, pp, rr)
        ctx.save_for_backward(xx, yy, pp, rr)
        ctx.lead = lead
        return out.reshape(*lead, n, H)

    @staticmethod
    def backward(ctx, grad_out):
        xx, yy, pp, rr = ctx.saved_tensors
        n, H = xx.shape[-2], xx.shape[-1]
        if grad_out.dtype != xx.dtype:
            raise TypeError(f"the output gradient must be {xx.dtype}, got {grad_out.dtype}")
        g = grad_out.reshape(-1, n, H).contiguous()
        gx, gy, gp, gr = binding.post_backward(g, xx, yy, pp, rr)
        lead = ctx.lead
        return (gx.reshape(*lead, n, H) if ctx.needs_input_grad[0] else None,
                gy.reshape(*lead, H) if ctx.needs_input_grad[1] else None,
                gp.reshape(*lead, n) if ctx.needs_input_grad[2] else None,
                gr.reshape(*lead, n, n) if ctx.needs_input_grad[3] else None)


def mhc_post(x: torch.Tensor, y: torch.Tensor, post: torch.Tensor, res: torch.Tensor) -> torch.Tensor:
    """Differentiable mHC post (see MhcPost)."""
    return MhcPost.apply(x, y, post, res)


class MhcPostSigmoid(torch.autograd.Function):
    """The mHC post with post = sigmoid(alpha * mix + b) computed inside the
    kernels ("perf: fuse mHC coefficient backward epilogue", Summary: the post
    sigmoid's derivative, grad_mix and the grad_b / alpha gradients).  The
    backward is one fused kernel for grad_x, grad_y, grad_res, grad_z and
    grad_mix, and one kernel summing grad_b and grad_alpha over tokens in a
    fixed order."""

    @staticmethod
    def forward(ctx, x, y, mix, alpha, b, res):
        if x.dtype not in (torch.bfloat16, torch.float16) or y.dtype != x.dtype:
            raise TypeError("expects x [...,n,H] and y [...,H] of one type, bf16 or f16")
        if mix.dtype != torch.float32 or res.dtype != torch.float32:
            raise TypeError("expects mix [...,n] and res [...,n,n] fp32")
        if x.dim() < 2:
            raise ValueError(f"x must be [...,n,H], got {tuple(x.shape)}")
        lead = x.shape[:-2]
        n, H = x.shape[-2], x.shape[-1]
        if y.shape != (*lead, H) or mix.shape != (*lead, n) or res.shape != (*lead, n, n):
            raise ValueError(f"shape mismatch: x {tuple(x.shape)}, y {tuple(y.shape)}, "
                             f"mix {tuple(mix.shape)}, res {tuple(res.shape)}")
        xx = x.reshape(-1, n, H).contiguous()
        yy = y.reshape(-1, H).contiguous()
        mm = mix.reshape(-1, n).contiguous()
        rr = res.reshape(-1, n, n).contiguous()
        a = alpha.reshape(1).contiguous()
        bb = b.contiguous()
        out = binding.post_sigmoid(xx, yy, mm, a, bb, rr)
        ctx.save_for_backward(xx, yy, mm, a, bb, rr)
        ctx.lead = lead
        ctx.alpha_shape = alpha.shape
        return out.reshape(*lead, n, H)

    @staticmethod
    def backward(ctx, grad_out):
        xx, yy, mm, a, bb, rr = ctx.saved_tensors
        n, H = xx.shape[-2], xx.shape[-1]
        if grad_out.dtype != xx.dtype:
            raise TypeError(f"the output gradient must be {xx.dtype}, got {grad_out.dtype}")
        g = grad_out.reshape(-1, n, H).contiguous()
        gx, gy, gz, gm, gr = binding.post_sigmoid_backward(g, xx, yy, mm, a, bb, rr)
        grad_alpha = grad_b = None
        if ctx.needs_input_grad[3] or ctx.needs_input_grad[4]:
            grad_b, grad_alpha = binding.sigmoid_param_grad(gz, mm)
            grad_alpha = grad_alpha.reshape(ctx.alpha_shape)
        lead = ctx.lead
        return (gx.reshape(*lead, n, H) if ctx.needs_input_grad[0] else None,
                gy.reshape(*lead, H) if ctx.needs_input_grad[1] else None,
                gm.reshape(*lead, n) if ctx.needs_input_grad[2] else None,
                grad_alpha if ctx.needs_input_grad[3] else None,
                grad_b if ctx.needs_input_grad[4] else None,
                gr.reshape(*lead, n, n) if ctx.needs_input_grad[5] else None)


def mhc_post_sigmoid(x: torch.Tensor, y: torch.Tensor, mix: torch.Tensor, alpha: torch.Tensor,
                     b: torch.Tensor, res: torch.Tensor) -> torch.Tensor:
    """Differentiable mHC post with post = sigmoid(alpha * mix + b) computed in the kernel."""
    return MhcPostSigmoid.apply(x, y, mix, alpha, b, res)

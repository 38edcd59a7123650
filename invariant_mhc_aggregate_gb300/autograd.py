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

Inputs may have any leading batch shape: ``residual [..., 4, H]`` and
``pre [..., 4]`` are flattened to tokens and the results reshaped back.
"""

from __future__ import annotations

import torch

from . import binding


class HAggregate(torch.autograd.Function):
    @staticmethod
    def forward(ctx, residual: torch.Tensor, pre: torch.Tensor) -> torch.Tensor:
        if residual.dtype != torch.bfloat16 or pre.dtype != torch.float32:
            raise TypeError("h_aggregate expects residual bf16 [...,4,H] and pre fp32 [...,4]")
        if residual.shape[:-1] != pre.shape or residual.shape[-2] != 4:
            raise ValueError(f"shape mismatch: residual {tuple(residual.shape)}, pre {tuple(pre.shape)}")
        lead = residual.shape[:-2]
        H = residual.shape[-1]
        r = residual.reshape(-1, 4, H).contiguous()
        p = pre.reshape(-1, 4).contiguous()
        out = binding.h_aggregate(r, p)
        ctx.save_for_backward(r, p)
        ctx.lead = lead
        return out.reshape(*lead, H)

    @staticmethod
    def backward(ctx, grad_out: torch.Tensor):
        r, p = ctx.saved_tensors
        H = r.shape[-1]
        if grad_out.dtype != torch.bfloat16:
            raise TypeError(f"the gradient of the bf16 output must be bf16, got {grad_out.dtype}")
        g = grad_out.reshape(-1, H).contiguous()
        grad_residual, grad_pre = binding.h_aggregate_backward(g, r, p)
        gr = grad_residual.reshape(*ctx.lead, 4, H) if ctx.needs_input_grad[0] else None
        gp = grad_pre.reshape(*ctx.lead, 4) if ctx.needs_input_grad[1] else None
        return gr, gp


def h_aggregate(residual: torch.Tensor, pre: torch.Tensor) -> torch.Tensor:
    """Differentiable batch-invariant H Aggregate (see the module docstring)."""
    return HAggregate.apply(residual, pre)

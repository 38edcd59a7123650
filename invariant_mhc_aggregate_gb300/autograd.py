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

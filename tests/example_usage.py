"""Usage example of the library (the one the README shows); run by
test_example_gpu.py on a GPU."""

import torch

from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.autograd import h_aggregate, mhc_post


def main():
    T, n, H = 4096, 4, 7168
    residual = torch.randn(T, n, H, device="cuda").to(torch.bfloat16).requires_grad_()
    pre = torch.rand(T, n, device="cuda", requires_grad=True)
    out = h_aggregate(residual, pre)                  # [T, H], one kernel
    out.float().square().mean().backward()            # residual.grad, pre.grad: one fused kernel

    # the same through the C ABI's names, into caller-owned buffers
    binding.mhc_h_aggregate_fwd(residual.detach(), pre.detach(), torch.empty_like(out))

    # the mHC post: out[t,k] = tree(res[t,k,j] * x[t,j]) + post[t,k] * y[t]
    x = torch.randn(T, n, H, device="cuda").to(torch.bfloat16)
    y = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    res = torch.softmax(torch.randn(T, n, n, device="cuda"), -1)
    streams = mhc_post(x, y, 2 * torch.rand(T, n, device="cuda"), res)   # [T, n, H]
    return out, residual.grad, pre.grad, streams


if __name__ == "__main__":
    main()

"""Run a number of steps of one of the library's call families on seeded
synthetic inputs, with nothing else in the process: a fixed workload for
profilers (``ncu -k ...``) and for quick timing.

    python -m invariant_mhc_aggregate_gb300.run_steps --family sigmoid --T 4096 --H 7168
    python -m invariant_mhc_aggregate_gb300.run_steps --family plain --H 7167 --steps 5

Families (one step = forward then backward):
  plain     mhc_aggregate_fwd / mhc_aggregate_bwd (pre given)
  sigmoid   mhc_aggregate_sigmoid_fwd / mhc_aggregate_sigmoid_bwd, then
            mhc_sigmoid_param_grad (pre computed from the mix)
  post      mhc_post_fwd / mhc_post_bwd (the layer output expanded onto the
            n streams)
  post_sigmoid
            mhc_post_sigmoid_fwd / mhc_post_sigmoid_bwd, then
            mhc_sigmoid_param_grad (post computed from the mix)

The buffers are PyTorch allocations (512-byte aligned), so the path follows
from H: H % 16 == 0 the 32-byte path, H % 8 == 0 the 16-byte path, even H
the 4-byte pair path, odd H the realigned 16-byte path.  ``--offset 2``
moves every BF16 buffer 2 bytes off its allocation (the realigned path for
any H >= 64).  Prints one line with the mean step time (CUDA events around
the steps, after one warm-up step).
"""

from __future__ import annotations

import argparse

import torch

from . import _build, binding
from .inputs import backward_inputs, coeff_inputs, post_inputs


def _shifted(t: torch.Tensor, offset: int) -> torch.Tensor:
    """A copy of t placed `offset` bytes past a 512-byte boundary."""
    if offset == 0:
        return t
    n = t.numel()
    buf = torch.empty(n + 256, dtype=t.dtype, device=t.device)
    view = buf[offset // t.element_size():offset // t.element_size() + n].view(t.shape)
    view.copy_(t)
    return view


def _time(step, steps: int) -> float:
    step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / steps


def _post(args, dev, dtype) -> None:
    T, H, n = args.T, args.H, args.n
    x, y, post, res, g = post_inputs(T, H, n, "normal", 6, device=dev, dtype=dtype, with_grad=True)
    x, y, g = (_shifted(t, args.offset) for t in (x, y, g))
    out = _shifted(torch.empty_like(x), args.offset)
    gx = _shifted(torch.empty_like(x), args.offset)
    gy = _shifted(torch.empty_like(y), args.offset)
    gp, gr = torch.empty_like(post), torch.empty_like(res)
    paths = (binding.PATH_NAMES[binding.post_fwd_path_raw(x.data_ptr(), y.data_ptr(), post.data_ptr(),
                                                           res.data_ptr(), out.data_ptr(), T, n, H)],
             binding.PATH_NAMES[binding.post_bwd_path_raw(*(t.data_ptr() for t in (g, x, y, post, res, gx,
                                                                                  gy, gp, gr)), T, n, H)])

    if args.family == "post":
        def step():
            binding.mhc_post_fwd(x, y, post, res, out)
            binding.mhc_post_bwd(g, x, y, post, res, gx, gy, gp, gr)
    else:
        mix, alpha, b = (t.to(dev) for t in coeff_inputs(T, n, "normal", 7))
        gm = torch.empty_like(mix)
        gb = torch.empty((n,), dtype=torch.float32, device=dev)
        ga = torch.empty((1,), dtype=torch.float32, device=dev)

        def step():
            binding.mhc_post_sigmoid_fwd(x, y, mix, alpha, b, res, out)
            binding.mhc_post_sigmoid_bwd(g, x, y, mix, alpha, b, res, gx, gy, gp, gm, gr)
            binding.mhc_sigmoid_param_grad(gp, mix, gb, ga)

    us = _time(step, args.steps)
    print(f"{args.family} T={T} H={H} n={n} {args.dtype} offset={args.offset} paths fwd/bwd={paths[0]}/"
          f"{paths[1]}: {us:.1f} us per step")


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--family", choices=("plain", "sigmoid", "post", "post_sigmoid"), default="plain")
    ap.add_argument("--T", type=int, default=4096)
    ap.add_argument("--H", type=int, default=7168)
    ap.add_argument("--n", type=int, default=4)
    ap.add_argument("--dtype", choices=("bf16", "f16"), default="bf16")
    ap.add_argument("--offset", type=int, default=0, help="byte offset of every 2-byte buffer (even)")
    ap.add_argument("--steps", type=int, default=3)
    args = ap.parse_args(argv)

    _build.build()
    binding.load()
    dev = torch.device("cuda", 0)
    dtype = torch.bfloat16 if args.dtype == "bf16" else torch.float16
    T, H, n = args.T, args.H, args.n
    if args.family in ("post", "post_sigmoid"):
        _post(args, dev, dtype)
        return
    g, res, pre = backward_inputs(T, H, "normal", 4, device=dev, n=n, dtype=dtype)
    g, res = _shifted(g, args.offset), _shifted(res, args.offset)
    out = _shifted(torch.empty((T, H), dtype=dtype, device=dev), args.offset)
    gres = _shifted(torch.empty((T, n, H), dtype=dtype, device=dev), args.offset)
    if args.family == "plain":
        grad_pre = torch.empty((T, n), dtype=torch.float32, device=dev)

        def step():
            binding.mhc_aggregate_fwd(res, pre, out)
            binding.mhc_aggregate_bwd(g, res, pre, gres, grad_pre)
    else:
        mix, alpha, b = (x.to(dev) for x in coeff_inputs(T, n, "normal", 5))
        grad_z = torch.empty((T, n), dtype=torch.float32, device=dev)
        grad_mix = torch.empty_like(grad_z)
        grad_b = torch.empty((n,), dtype=torch.float32, device=dev)
        grad_alpha = torch.empty((1,), dtype=torch.float32, device=dev)

        def step():
            binding.mhc_aggregate_sigmoid_fwd(res, mix, alpha, b, out)
            binding.mhc_aggregate_sigmoid_bwd(g, res, mix, alpha, b, gres, grad_z, grad_mix)
            binding.mhc_sigmoid_param_grad(grad_z, mix, grad_b, grad_alpha)

    gp = grad_pre if args.family == "plain" else grad_z
    coef = pre if args.family == "plain" else mix
    paths = (binding.PATH_NAMES[binding.agg_fwd_path_raw(res.data_ptr(), coef.data_ptr(), out.data_ptr(),
                                                          T, n, H)],
             binding.PATH_NAMES[binding.agg_bwd_path_raw(g.data_ptr(), res.data_ptr(), coef.data_ptr(),
                                                          gres.data_ptr(), gp.data_ptr(), T, n, H)])
    step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    print(f"{args.family} T={T} H={H} n={n} {args.dtype} offset={args.offset} paths fwd/bwd={paths[0]}/"
          f"{paths[1]}: {e0.elapsed_time(e1) * 1e3 / args.steps:.1f} us per step")


if __name__ == "__main__":
    main()

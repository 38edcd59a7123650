"""Seeded synthetic inputs for the mHC pre "H Aggregate" workloads.

This module only draws random numbers; it holds none of the operation's
arithmetic, and both the CUDA path and the CPU oracle are fed from it.

The pages measure no dataset: their workloads are (T, H) shapes of a BF16
residual ``[T,4,H]`` and an FP32 ``pre`` ``[T,4]`` ("Add batch-invariant
h_aggregate kernel", Summary and the Performance table).  The value recipes
below are this library's stand-ins for them:

==============  =====================================================================
recipe          values
==============  =====================================================================
``normal``      residual ~ N(0,1) rounded to BF16 (RNE); pre ~ U(0,1)
``ragged``      as ``normal``; then 5% of pre entries set to exactly 0.0 and 5% to
                exactly 1.0
``decode``      residual ~ 2*N(0,1), each entry scaled by 100 with probability 1%,
                then rounded to BF16; pre = sigmoid(N(0,1))
backward ``g``  g ~ N(0,1) rounded to BF16, drawn after residual and pre
==============  =====================================================================

For the pre coefficients computed from the mix (``coeff_inputs``): ``mix``
``[T,n]`` FP32, ``alpha`` ``[1]`` and ``b`` ``[n]``:

==============  =====================================================================
``normal``      mix ~ N(0,1); alpha ~ U(0.5, 2); b ~ 0.5*N(0,1)
``wide``        mix ~ 16*N(0,1), then 5% of entries set to exactly 0.0 and 2% to
                +-100 (sigmoid saturates, 1 - sigmoid underflows toward the
                subnormal range); alpha and b as ``normal``
==============  =====================================================================

For the mHC post (``post_inputs``): ``x`` ``[T,n,H]`` (the streams), ``y``
``[T,H]`` (the layer output), ``post`` ``[T,n]`` and ``res`` ``[T,n,n]`` FP32,
and for the backward ``g`` ``[T,n,H]``:

==============  =====================================================================
``normal``      x, y, g ~ N(0,1) rounded to the storage type; post ~ 2*U(0,1); each
                row of res = exp(N(0,1)) divided by its row sum (rows of positive
                mixing weights near a unit sum)
``ragged``      as ``normal``; then 10% of tokens get res = the identity and 5% of
                post entries exactly 0.0
==============  =====================================================================

Every draw comes from one ``torch.Generator`` seeded with the workload's seed,
in a fixed order (residual, pre, masks, g), so a (recipe, T, H, seed, device)
tuple always gives the same bytes on a given PyTorch build.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

RECIPES = ("normal", "ragged", "decode")
COEFF_RECIPES = ("normal", "wide")


@dataclass(frozen=True)
class Workload:
    """One named workload: its shapes, value recipe and seed."""

    name: str
    direction: str            # "fwd" or "bwd"
    shapes: tuple             # tuple of (T, H)
    recipe: str
    seed: int
    note: str = ""


#: The five workloads the library is checked and measured on.
WORKLOADS = (
    Workload("fwd_t129_h4096", "fwd", ((129, 4096),), "normal", 0,
             "bit-exact vs the oracle; full batch vs 129 one-token calls"),
    Workload("fwd_ragged", "fwd", ((3, 1279), (1, 4097), (17, 2050)), "ragged", 1,
             "odd-H scalar tail and ragged shapes"),
    Workload("fwd_decode", "fwd", ((1, 4096), (8, 4096), (128, 4096),
                                   (1, 7168), (8, 7168), (128, 7168)), "decode", 2,
             "decode-sized latency sweep"),
    Workload("fwd_prefill", "fwd", ((1024, 7168), (4096, 7168), (16384, 7168),
                                    (65536, 7168)), "normal", 3,
             "bandwidth-bound prefill"),
    Workload("bwd_t4096_h7168", "bwd", ((4096, 7168),), "normal", 4,
             "fused grad_residual + grad_pre"),
)


def workload(name: str) -> Workload:
    for w in WORKLOADS:
        if w.name == name:
            return w
    raise KeyError(name)


def _generator(device, seed: int) -> torch.Generator:
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(int(seed))
    return gen


def forward_inputs(T: int, H: int, recipe: str = "normal", seed: int = 0,
                   device="cpu", n: int = 4,
                   dtype=torch.bfloat16) -> tuple[torch.Tensor, torch.Tensor]:
    """(residual [T,n,H] in `dtype`, pre fp32 [T,n]) drawn on ``device``."""
    gen = _generator(device, seed)
    return _draw_forward(T, H, recipe, gen, device, n, dtype)


def backward_inputs(T: int, H: int, recipe: str = "normal", seed: int = 4,
                    device="cpu", n: int = 4,
                    dtype=torch.bfloat16) -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(g [T,H], residual [T,n,H], pre fp32 [T,n]) drawn on ``device``; g and the
    residual in `dtype` (bfloat16 or float16, rounded to nearest even)."""
    gen = _generator(device, seed)
    residual, pre = _draw_forward(T, H, recipe, gen, device, n, dtype)
    g = torch.randn((T, H), generator=gen, device=device, dtype=torch.float32)
    return g.to(dtype), residual, pre


def coeff_inputs(T: int, n: int = 4, recipe: str = "normal", seed: int = 5,
                 device="cpu") -> tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(mix fp32 [T,n], alpha fp32 [1], b fp32 [n]) drawn on ``device``."""
    if recipe not in COEFF_RECIPES:
        raise ValueError(f"unknown recipe {recipe!r}; expected one of {COEFF_RECIPES}")
    gen = _generator(device, seed)
    f32 = torch.float32
    mix = torch.randn((T, n), generator=gen, device=device, dtype=f32)
    alpha = 0.5 + 1.5 * torch.rand((1,), generator=gen, device=device, dtype=f32)
    b = 0.5 * torch.randn((n,), generator=gen, device=device, dtype=f32)
    if recipe == "wide":
        mix.mul_(16.0)
        u = torch.rand((T, n), generator=gen, device=device, dtype=f32)
        sign = torch.where(torch.rand((T, n), generator=gen, device=device, dtype=f32) < 0.5,
                           -1.0, 1.0)
        mix = torch.where(u < 0.05, torch.zeros_like(mix), mix)
        mix = torch.where((u >= 0.05) & (u < 0.07), 100.0 * sign, mix)
    return mix.contiguous(), alpha, b


POST_RECIPES = ("normal", "ragged")


def post_inputs(T: int, H: int, n: int = 4, recipe: str = "normal", seed: int = 6,
                device="cpu", dtype=torch.bfloat16, with_grad: bool = False):
    """(x [T,n,H], y [T,H], post fp32 [T,n], res fp32 [T,n,n]) drawn on ``device``,
    then g [T,n,H] when ``with_grad``; x, y and g in `dtype`."""
    if recipe not in POST_RECIPES:
        raise ValueError(f"unknown recipe {recipe!r}; expected one of {POST_RECIPES}")
    gen = _generator(device, seed)
    f32 = torch.float32
    x = torch.randn((T, n, H), generator=gen, device=device, dtype=f32).to(dtype)
    y = torch.randn((T, H), generator=gen, device=device, dtype=f32).to(dtype)
    post = 2.0 * torch.rand((T, n), generator=gen, device=device, dtype=f32)
    w = torch.exp(torch.randn((T, n, n), generator=gen, device=device, dtype=f32))
    res = w / w.sum(dim=-1, keepdim=True)
    if recipe == "ragged":
        ident = torch.rand((T,), generator=gen, device=device, dtype=f32) < 0.10
        eye = torch.eye(n, device=device, dtype=f32).expand(T, n, n)
        res = torch.where(ident[:, None, None], eye, res)
        zero = torch.rand((T, n), generator=gen, device=device, dtype=f32) < 0.05
        post = torch.where(zero, torch.zeros_like(post), post)
    out = [x.contiguous(), y.contiguous(), post.contiguous(), res.contiguous()]
    if with_grad:
        out.append(torch.randn((T, n, H), generator=gen, device=device, dtype=f32).to(dtype))
    return tuple(out)


def _draw_forward(T, H, recipe, gen, device, n=4, dtype=torch.bfloat16):
    if recipe not in RECIPES:
        raise ValueError(f"unknown recipe {recipe!r}; expected one of {RECIPES}")
    f32 = torch.float32
    r = torch.randn((T, n, H), generator=gen, device=device, dtype=f32)
    if recipe == "decode":
        r.mul_(2.0)
        outlier = torch.rand((T, n, H), generator=gen, device=device, dtype=f32) < 0.01
        r = torch.where(outlier, r * 100.0, r)
        pre = torch.sigmoid(torch.randn((T, n), generator=gen, device=device, dtype=f32))
    else:
        pre = torch.rand((T, n), generator=gen, device=device, dtype=f32)
        if recipe == "ragged":
            u = torch.rand((T, n), generator=gen, device=device, dtype=f32)
            pre = torch.where(u < 0.05, torch.zeros_like(pre), pre)
            pre = torch.where((u >= 0.05) & (u < 0.10), torch.ones_like(pre), pre)
    residual = r.to(dtype)
    del r
    return residual.contiguous(), pre.contiguous()


def as_u16(x: torch.Tensor):
    """BF16 / FP16 tensor -> numpy uint16 bit patterns (host copy)."""
    return x.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")


def as_f32(x: torch.Tensor):
    """FP32 tensor -> numpy float32 (host copy)."""
    return x.detach().contiguous().cpu().numpy()

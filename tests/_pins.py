"""Checks that pin the CPU oracle to facts outside itself.

Each ``check_*`` function takes an ``oracle.Oracle`` and raises
``AssertionError`` when the oracle disagrees with a hand-worked value from
``tests/golden``, an independent library routine, exact rational arithmetic, a
closed-form error bound or an exact invariant.  ``test_oracle_pins.py`` runs
them on the real oracle; ``test_oracle_mutants.py`` runs them on copies of the
oracle with planted mistakes and expects every mistake to be caught.

Sources: "Add batch-invariant h_aggregate kernel" (Summary formula, Batch
invariance rules) for the forward; the same page's reviewer request for the
backward, whose formula here is the derivative of the Summary formula.
"""

from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U = 2.0 ** -24  # unit roundoff of binary32


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def golden_rows(name: str):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def f32_from_bits(u: int) -> np.float32:
    return np.array([u], dtype=np.uint32).view(np.float32)[0]


def f32_bits(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).view(np.uint32)


def bf16_widen(u16: np.ndarray) -> np.ndarray:
    """BF16 patterns -> float32, by shifting into the upper half (independent of the oracle)."""
    return (np.asarray(u16, dtype=np.uint32) << 16).view(np.float32)


def round_rne(x: Fraction, p: int, emin: int = -126, emax: int = 127) -> float:
    """Round a rational to a binary format with p significant bits, exponent range
    [emin, emax], ties to even, subnormals kept, overflow to infinity.  The result
    is returned as a Python float (exact for binary32 and BF16 values)."""
    if x == 0:
        return 0.0
    sign = -1.0 if x < 0 else 1.0
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    quantum = Fraction(2) ** (e - p + 1)
    m = a / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    r = fl * quantum
    if r >= Fraction(2) ** (emax + 1):
        return sign * math.inf
    return sign * float(r)


def exact_mul(a: float, b: float) -> float:
    """One binary32 multiply, rounded to nearest even, by exact rationals."""
    if a == 0.0 or b == 0.0:
        return math.copysign(0.0, math.copysign(1.0, a) * math.copysign(1.0, b))
    return round_rne(Fraction(a) * Fraction(b), 24)


def exact_add(a: float, b: float) -> float:
    """One binary32 add, rounded to nearest even, by exact rationals (IEEE zero signs)."""
    if math.isinf(a) or math.isinf(b):
        return a + b
    s = Fraction(a) + Fraction(b)
    if s == 0:
        both_neg = math.copysign(1.0, a) < 0 and math.copysign(1.0, b) < 0
        return -0.0 if both_neg else 0.0
    return round_rne(s, 24)


def to_bf16_exact(x: float) -> float:
    if math.isinf(x) or x == 0.0:
        return x
    return round_rne(Fraction(x), 8)


def bf16_bits_of(x: float) -> int:
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0] >> 16)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of BF16 values at |x| (8 significant bits), for finite x."""
    ax = np.abs(x.astype(np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def random_bf16(rng, shape, scale=1.0) -> np.ndarray:
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    bits = x.view(np.uint32)
    # truncate-and-round by numpy integer arithmetic on the pattern (test-local RNE)
    kept = bits >> 16
    dropped = bits & 0xFFFF
    up = (dropped > 0x8000) | ((dropped == 0x8000) & ((kept & 1) == 1))
    return (kept + up).astype(np.uint16)


# --------------------------------------------------------------------------
# BF16 conversion
# --------------------------------------------------------------------------

def check_bf16_golden(o):
    for fbits, bbits, *_ in golden_rows("bf16_rounding.txt"):
        x = f32_from_bits(int(fbits, 16))
        got = int(o.bf16_from_float(np.array([x], dtype=np.float32))[0])
        assert got == int(bbits, 16), f"bf16({fbits}) = {got:04X}, expected {bbits}"


def check_bf16_roundtrip_exhaustive(o):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    wide = o.float_from_bf16(pats)
    assert np.array_equal(f32_bits(wide), pats.astype(np.uint32) << 16)
    back = o.bf16_from_float(wide)
    nan = ((pats & 0x7F80) == 0x7F80) & ((pats & 0x007F) != 0)
    assert np.array_equal(back[~nan], pats[~nan])
    # NaNs stay NaN (payload not part of the contract)
    assert np.all(((back[nan] & 0x7F80) == 0x7F80) & ((back[nan] & 0x007F) != 0))


def check_bf16_vs_torch(o):
    import torch
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    # add every pattern near each BF16 rounding boundary in a few binades
    base = np.arange(0x3F000000, 0x3F000000 + (1 << 18), dtype=np.uint32)
    edges = np.concatenate([bits, base, base | 0x80000000, np.arange(0, 1 << 16, dtype=np.uint32),
                            np.array([0x7F7FFFFF, 0x7F7F8000, 0xFF7F8000], dtype=np.uint32)])
    x = edges.view(np.float32)
    finite = np.isfinite(x)
    x = x[finite]
    ours = o.bf16_from_float(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches vs torch, e.g. {x[bad[:4]].view(np.uint32)}"


def check_widen_vs_torch(o):
    import torch
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = o.float_from_bf16(pats)
    ref = torch.from_numpy(pats.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    finite = np.isfinite(ref)
    assert np.array_equal(f32_bits(ours)[finite], f32_bits(ref)[finite])
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------

def _fwd_cases():
    for name, r0, r1, r2, r3, p0, p1, p2, p3, out in golden_rows("fwd_worked_examples.txt"):
        r = np.array([int(v, 16) for v in (r0, r1, r2, r3)], dtype=np.uint16)
        pre = np.array([f32_from_bits(int(v, 16)) for v in (p0, p1, p2, p3)], dtype=np.float32)
        yield name, r, pre, int(out, 16)


def check_fwd_golden(o):
    rng = np.random.default_rng(11)
    for name, r, pre, expected in _fwd_cases():
        got = int(o.fwd(r.reshape(1, 4, 1), pre.reshape(1, 4))[0, 0])
        assert got == expected, f"{name}: {got:04X} != {expected:04X}"
        # the same element inside a larger ragged batch, at token 2, position 5
        T, H = 4, 13
        res = random_bf16(rng, (T, 4, H))
        pr = rng.random((T, 4), dtype=np.float32)
        res[2, :, 5] = r
        pr[2] = pre
        got = int(o.fwd(res, pr)[2, 5])
        assert got == expected, f"{name} (embedded): {got:04X} != {expected:04X}"


def _fwd_exact(r_u16, pre):
    r = bf16_widen(r_u16)
    T, _, H = r.shape
    out = np.empty((T, H), dtype=np.uint16)
    for t in range(T):
        for h in range(H):
            p = [exact_mul(float(pre[t, k]), float(r[t, k, h])) for k in range(4)]
            s = exact_add(exact_add(p[0], p[1]), exact_add(p[2], p[3]))
            out[t, h] = bf16_bits_of(to_bf16_exact(s))
    return out


def check_fwd_exact_rational(o):
    rng = np.random.default_rng(12)
    # full-precision values
    res = random_bf16(rng, (3, 4, 37))
    pre = rng.random((3, 4), dtype=np.float32)
    assert np.array_equal(o.fwd(res, pre), _fwd_exact(res, pre))
    # coarse values: products and sums land on rounding ties often
    res = random_bf16(rng, (4, 4, 40), scale=4.0)
    res &= np.uint16(0xFFF0)  # 3 fraction bits
    pre = (rng.integers(1, 1 << 12, size=(4, 4)) * 2.0 ** -9).astype(np.float32)
    pre[0, 1] = 1.0 + 2.0 ** -8
    assert np.array_equal(o.fwd(res, pre), _fwd_exact(res, pre))


def check_fwd_fp64_bound(o):
    rng = np.random.default_rng(13)
    res = random_bf16(rng, (64, 4, 515))
    pre = rng.random((64, 4), dtype=np.float32)
    out = bf16_widen(o.fwd(res, pre)).astype(np.float64)
    prod = pre.astype(np.float64)[:, :, None] * bf16_widen(res).astype(np.float64)  # exact
    exact = prod.sum(axis=1)
    mag = np.abs(prod).sum(axis=1)
    bound = 0.5 * bf16_ulp(out) + 3.01 * U * mag
    err = np.abs(out - exact)
    assert np.all(err <= bound), f"max excess {np.max(err - bound)}"


def check_fwd_one_hot(o):
    rng = np.random.default_rng(14)
    res = random_bf16(rng, (6, 4, 77))
    res[res == 0x8000] = 0  # -0 may come out as +0 by IEEE rules
    for k in range(4):
        pre = np.zeros((6, 4), dtype=np.float32)
        pre[:, k] = 1.0
        out = o.fwd(res, pre)
        assert np.array_equal(out, res[:, k, :]), f"one-hot k={k}"


def check_fwd_zero_pre(o):
    rng = np.random.default_rng(15)
    res = random_bf16(rng, (5, 4, 33))
    out = o.fwd(res, np.zeros((5, 4), dtype=np.float32))
    assert np.all((out == 0) | (out == 0x8000))


def check_fwd_symmetries(o):
    """The (0+1)+(2+3) tree is unchanged by swapping 0<->1, 2<->3 or the two pairs."""
    rng = np.random.default_rng(16)
    res = random_bf16(rng, (8, 4, 301))
    res &= np.uint16(0xFFF8)
    pre = (rng.integers(1, 1 << 14, size=(8, 4)) * 2.0 ** -13).astype(np.float32)
    base = o.fwd(res, pre)
    for perm in ([1, 0, 2, 3], [0, 1, 3, 2], [2, 3, 0, 1], [3, 2, 1, 0]):
        assert np.array_equal(o.fwd(res[:, perm, :], pre[:, perm]), base), f"perm {perm}"


def check_fwd_scaling(o):
    rng = np.random.default_rng(17)
    res = random_bf16(rng, (4, 4, 99))
    pre = rng.random((4, 4), dtype=np.float32) + 0.5
    base = bf16_widen(o.fwd(res, pre))
    for e in (-3, 1, 5):
        scaled = bf16_widen(o.fwd(res, (pre * np.float32(2.0 ** e)).astype(np.float32)))
        assert np.array_equal(scaled, base * np.float32(2.0 ** e)), f"scale 2^{e}"


def check_fwd_negation(o):
    rng = np.random.default_rng(18)
    res = random_bf16(rng, (4, 4, 64))
    pre = rng.random((4, 4), dtype=np.float32)
    a = bf16_widen(o.fwd(res, pre))
    b = bf16_widen(o.fwd(res, -pre))
    assert np.array_equal(a, -b)


def check_fwd_token_independent(o):
    rng = np.random.default_rng(19)
    res = random_bf16(rng, (9, 4, 21))
    pre = rng.random((9, 4), dtype=np.float32)
    full = o.fwd(res, pre)
    for t in range(9):
        assert np.array_equal(o.fwd(res[t:t + 1], pre[t:t + 1])[0], full[t])


# --------------------------------------------------------------------------
# backward: grad_residual
# --------------------------------------------------------------------------

def check_gr_golden(o):
    rng = np.random.default_rng(21)
    for name, pbits, gbits, ebits in golden_rows("grad_residual_worked_examples.txt"):
        pre_v = f32_from_bits(int(pbits, 16))
        T, H = 3, 11
        g = random_bf16(rng, (T, H))
        pre = rng.random((T, 4), dtype=np.float32)
        g[1, 7] = int(gbits, 16)
        pre[1, 2] = pre_v
        got = int(o.grad_residual(g, pre)[1, 2, 7])
        assert got == int(ebits, 16), f"{name}: {got:04X} != {ebits}"


def check_gr_exact_rational(o):
    rng = np.random.default_rng(22)
    g = random_bf16(rng, (3, 29))
    pre = rng.random((3, 4), dtype=np.float32) * np.float32(3.0)
    got = o.grad_residual(g, pre)
    gw = bf16_widen(g)
    for t in range(3):
        for k in range(4):
            for h in range(29):
                v = to_bf16_exact(exact_mul(float(pre[t, k]), float(gw[t, h])))
                assert got[t, k, h] == bf16_bits_of(v), (t, k, h)


def check_gr_identity_onehot(o):
    rng = np.random.default_rng(23)
    g = random_bf16(rng, (5, 40))
    pre = np.zeros((5, 4), dtype=np.float32)
    pre[:, 2] = 1.0
    pre[:, 0] = 4.0
    pre[:, 3] = 0.5
    got = o.grad_residual(g, pre)
    gw = bf16_widen(g)
    assert np.array_equal(got[:, 2, :], g)
    assert np.array_equal(bf16_widen(got[:, 0, :]), gw * np.float32(4.0))
    assert np.array_equal(bf16_widen(got[:, 3, :]), gw * np.float32(0.5))
    assert np.all(bf16_widen(got[:, 1, :]) == 0.0)


# --------------------------------------------------------------------------
# backward: grad_pre
# --------------------------------------------------------------------------

def check_gp_golden(o):
    for name, H, k, carrier, positions, expected in golden_rows("grad_pre_order_cases.txt"):
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
        got = f32_bits(o.grad_pre(g, res))[0]
        want = np.zeros(4, dtype=np.uint32)
        want[k] = int(expected, 16)
        assert np.array_equal(got, want), f"{name}: {[hex(v) for v in got]} != {[hex(v) for v in want]}"


def check_gp_integer_exact(o):
    """Integer-valued g and r with every partial sum below 2^24: any order gives the
    exact integer sum, which fixes products, lane coverage, padding and rows."""
    rng = np.random.default_rng(24)
    for H in (1, 7, 8, 9, 255, 2047, 2048, 2049, 4104, 7168, 9001):
        T = 3
        gi = rng.integers(-8, 9, size=(T, H))
        ri = rng.integers(-8, 9, size=(T, 4, H))
        g = np.array([bf16_bits_of(float(v)) for v in range(-8, 9)], dtype=np.uint16)[gi + 8]
        r = np.array([bf16_bits_of(float(v)) for v in range(-8, 9)], dtype=np.uint16)[ri + 8]
        got = o.grad_pre(g, r)
        want = np.einsum("th,tkh->tk", gi, ri).astype(np.float64)
        assert np.array_equal(got.astype(np.float64), want), f"H={H}"


def order256_depth(H: int) -> int:
    """Longest chain of binary32 adds any product goes through in ORDER-256."""
    C = (H + 7) // 8
    return 3 + (C + 255) // 256 + 5 + 3


def check_gp_fp64_bound(o):
    rng = np.random.default_rng(25)
    for H in (8, 1279, 4097, 7168):
        T = 4
        g = random_bf16(rng, (T, H))
        r = random_bf16(rng, (T, 4, H))
        got = o.grad_pre(g, r).astype(np.float64)
        q = bf16_widen(g).astype(np.float64)[:, None, :] * bf16_widen(r).astype(np.float64)
        exact = np.array([[math.fsum(q[t, k]) for k in range(4)] for t in range(T)])
        mag = np.abs(q).sum(axis=2)
        bound = 1.01 * order256_depth(H) * U * mag
        assert np.all(np.abs(got - exact) <= bound), f"H={H}"


ALL_CHECKS = [
    check_bf16_golden,
    check_bf16_roundtrip_exhaustive,
    check_bf16_vs_torch,
    check_widen_vs_torch,
    check_fwd_golden,
    check_fwd_exact_rational,
    check_fwd_fp64_bound,
    check_fwd_one_hot,
    check_fwd_zero_pre,
    check_fwd_symmetries,
    check_fwd_scaling,
    check_fwd_negation,
    check_fwd_token_independent,
    check_gr_golden,
    check_gr_exact_rational,
    check_gr_identity_onehot,
    check_gp_golden,
    check_gp_integer_exact,
    check_gp_fp64_bound,
]


# --------------------------------------------------------------------------
# FP16 storage and the general stream count (a reading beyond the pages)
# --------------------------------------------------------------------------

def f16_widen(u16: np.ndarray) -> np.ndarray:
    """binary16 patterns -> float32 through numpy's own float16 (independent of the oracle)."""
    return np.asarray(u16, dtype=np.uint16).view(np.float16).astype(np.float32)


def to_f16_exact(x: float) -> float:
    if math.isinf(x) or x == 0.0:
        return x
    return round_rne(Fraction(x), 11, emin=-14, emax=15)


def f16_bits_of(x: float) -> int:
    return int(np.array([x], dtype=np.float16).view(np.uint16)[0])


STORAGE = {
    "bf16": (bf16_widen, to_bf16_exact, bf16_bits_of),
    "f16": (f16_widen, to_f16_exact, f16_bits_of),
}


def random_f16(rng, shape, scale=1.0) -> np.ndarray:
    return (rng.standard_normal(shape) * scale).astype(np.float16).view(np.uint16)


def random_storage(rng, shape, dtype, scale=1.0):
    return random_bf16(rng, shape, scale) if dtype == "bf16" else random_f16(rng, shape, scale)


def check_f16_golden(o):
    for fbits, hbits, *_ in golden_rows("f16_rounding.txt"):
        x = f32_from_bits(int(fbits, 16))
        got = int(o.f16_from_float(np.array([x], dtype=np.float32))[0])
        assert got == int(hbits, 16), f"f16({fbits}) = {got:04X}, expected {hbits}"


def check_f16_roundtrip_exhaustive(o):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    wide = o.float_from_f16(pats)
    ref = pats.view(np.float16).astype(np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(f32_bits(wide)[finite], f32_bits(ref)[finite])
    assert np.array_equal(np.isnan(wide), np.isnan(ref))
    back = o.f16_from_float(wide)
    nan = ((pats & 0x7C00) == 0x7C00) & ((pats & 0x03FF) != 0)
    assert np.array_equal(back[~nan], pats[~nan])
    assert np.all(((back[nan] & 0x7C00) == 0x7C00) & ((back[nan] & 0x03FF) != 0))


def check_f16_vs_torch(o):
    import torch
    rng = np.random.default_rng(8)
    bits = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    base = np.arange(0x33000000, 0x33000000 + (1 << 18), dtype=np.uint32)        # subnormal range
    near_one = np.arange(0x3F7E0000, 0x3F7E0000 + (1 << 18), dtype=np.uint32)
    near_max = np.arange(0x477F0000, 0x477F0000 + (1 << 17), dtype=np.uint32)
    x = np.concatenate([bits, base, near_one, near_max, near_max | 0x80000000]).view(np.float32)
    x = x[np.isfinite(x)]
    ours = o.f16_from_float(x)
    ref = torch.from_numpy(x.copy()).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches vs torch, e.g. {x[bad[:4]].view(np.uint32)}"


def _hc_cases():
    for row in golden_rows("fwd_hc_worked_examples.txt"):
        name, dtype, n = row[0], row[1], int(row[2])
        r = np.array([int(v, 16) for v in row[3:3 + n]], dtype=np.uint16)
        pre = np.array([f32_from_bits(int(v, 16)) for v in row[3 + n:3 + 2 * n]], dtype=np.float32)
        yield name, dtype, n, r, pre, int(row[3 + 2 * n], 16)


def check_agg_golden(o):
    rng = np.random.default_rng(51)
    for name, dtype, n, r, pre, expected in _hc_cases():
        got = int(o.aggregate_fwd(r.reshape(1, n, 1), pre.reshape(1, n), dtype)[0, 0])
        assert got == expected, f"{name}: {got:04X} != {expected:04X}"
        T, H = 3, 11
        res = random_storage(rng, (T, n, H), dtype)
        pr = rng.random((T, n), dtype=np.float32)
        res[1, :, 4] = r
        pr[1] = pre
        got = int(o.aggregate_fwd(res, pr, dtype)[1, 4])
        assert got == expected, f"{name} (embedded): {got:04X} != {expected:04X}"


def check_agg_n4_bf16_is_the_pages_op(o):
    rng = np.random.default_rng(52)
    res = random_bf16(rng, (5, 4, 77))
    pre = rng.random((5, 4), dtype=np.float32)
    g = random_bf16(rng, (5, 77))
    assert np.array_equal(o.aggregate_fwd(res, pre, "bf16"), o.fwd(res, pre))
    gr1, gp1 = o.aggregate_bwd(g, res, pre, "bf16")
    gr2, gp2 = o.bwd(g, res, pre)
    assert np.array_equal(gr1, gr2) and np.array_equal(f32_bits(gp1), f32_bits(gp2))


def _agg_exact(r_u16, pre, dtype):
    widen, rnd, bits = STORAGE[dtype]
    r = widen(r_u16)
    T, n, H = r.shape
    out = np.empty((T, H), dtype=np.uint16)
    for t in range(T):
        for h in range(H):
            p = [exact_mul(float(pre[t, k]), float(r[t, k, h])) for k in range(n)]
            while len(p) > 1:
                p = [exact_add(p[2 * i], p[2 * i + 1]) for i in range(len(p) // 2)]
            out[t, h] = bits(rnd(p[0]))
    return out


def check_agg_exact_rational(o):
    rng = np.random.default_rng(53)
    for dtype in ("bf16", "f16"):
        for n in (1, 2, 4, 8):
            res = random_storage(rng, (2, n, 13), dtype, scale=3.0)
            pre = rng.random((2, n), dtype=np.float32) * np.float32(2.0)
            assert np.array_equal(o.aggregate_fwd(res, pre, dtype), _agg_exact(res, pre, dtype)), (dtype, n)
        # coarse values: ties in the final rounding are frequent
        res = random_storage(rng, (3, 8, 16), dtype, scale=4.0)
        res &= np.uint16(0xFFF0 if dtype == "bf16" else 0xFF80)
        pre = (rng.integers(1, 1 << 12, size=(3, 8)) * 2.0 ** -9).astype(np.float32)
        assert np.array_equal(o.aggregate_fwd(res, pre, dtype), _agg_exact(res, pre, dtype)), dtype


def check_agg_one_hot(o):
    rng = np.random.default_rng(54)
    for dtype in ("bf16", "f16"):
        for n in (1, 2, 8):
            res = random_storage(rng, (4, n, 33), dtype)
            res[res == 0x8000] = 0
            for k in range(n):
                pre = np.zeros((4, n), dtype=np.float32)
                pre[:, k] = 1.0
                assert np.array_equal(o.aggregate_fwd(res, pre, dtype), res[:, k, :]), (dtype, n, k)


def check_agg_grad_residual_exact(o):
    rng = np.random.default_rng(55)
    for dtype in ("bf16", "f16"):
        widen, rnd, bits = STORAGE[dtype]
        for n in (1, 2, 8):
            g = random_storage(rng, (2, 9), dtype)
            res = random_storage(rng, (2, n, 9), dtype)
            pre = rng.random((2, n), dtype=np.float32) * np.float32(3.0)
            gr, _ = o.aggregate_bwd(g, res, pre, dtype)
            gw = widen(g)
            for t in range(2):
                for k in range(n):
                    for h in range(9):
                        want = bits(rnd(exact_mul(float(pre[t, k]), float(gw[t, h]))))
                        assert gr[t, k, h] == want, (dtype, n, t, k, h)


def check_agg_grad_pre_integer_exact(o):
    rng = np.random.default_rng(56)
    for dtype in ("bf16", "f16"):
        _, _, bits = STORAGE[dtype]
        lut = np.array([bits(float(v)) for v in range(-8, 9)], dtype=np.uint16)
        for n, H in ((1, 9), (2, 2049), (8, 4104), (8, 13)):
            gi = rng.integers(-8, 9, size=(2, H))
            ri = rng.integers(-8, 9, size=(2, n, H))
            _, gp = o.aggregate_bwd(lut[gi + 8], lut[ri + 8], np.ones((2, n), dtype=np.float32), dtype)
            assert np.array_equal(gp.astype(np.float64), np.einsum("th,tkh->tk", gi, ri).astype(np.float64)), (dtype, n, H)


def check_agg_grad_pre_order_f16(o):
    """The ORDER-256 golden cases with FP16 storage (1 = 0x3C00, 2^-24 = 0x0001,
    -0 = 0x8000), in an n = 8 layout."""
    remap = {0x3F80: 0x3C00, 0x3380: 0x0001, 0x8000: 0x8000}
    for name, H, k, carrier, positions, expected in golden_rows("grad_pre_order_cases.txt"):
        H, k = int(H), int(k)
        vals = np.zeros(H, dtype=np.uint16)
        for item in positions.split(","):
            pos, v = item.split(":")
            if pos == "*":
                vals[:] = remap[int(v, 16)]
            else:
                vals[int(pos)] = remap[int(v, 16)]
        n = 8
        g = np.full((1, H), 0x3C00, dtype=np.uint16)
        res = np.zeros((1, n, H), dtype=np.uint16)
        kk = k + 4
        if carrier == "r":
            res[0, kk] = vals
        else:
            g[0] = vals
            res[0, kk] = 0x3C00
        _, gp = o.aggregate_bwd(g, res, np.ones((1, n), dtype=np.float32), "f16")
        want = np.zeros(n, dtype=np.uint32)
        want[kk] = int(expected, 16)
        assert np.array_equal(f32_bits(gp)[0], want), name


def check_fwd_fp64_emulation(o):
    """FP64 brute force on tiny shapes: each binary32 operation computed in FP64
    and rounded once to binary32 is correctly rounded (53 >= 2*24 + 2, so the
    double rounding is innocuous), and the final BF16 rounding is numpy's own
    RNE on the pattern; every element must match."""
    rng = np.random.default_rng(57)
    for T, H in ((1, 1), (2, 7), (3, 64)):
        res = random_bf16(rng, (T, 4, H), scale=2.0)
        pre = rng.random((T, 4), dtype=np.float32)
        r = bf16_widen(res).astype(np.float64)
        p = pre.astype(np.float64)
        f32 = lambda x: np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
        prod = [f32(p[:, k, None] * r[:, k, :]) for k in range(4)]
        s = f32(f32(prod[0] + prod[1]) + f32(prod[2] + prod[3])).astype(np.float32)
        bits = s.view(np.uint32)
        kept = bits >> 16
        dropped = bits & 0xFFFF
        up = (dropped > 0x8000) | ((dropped == 0x8000) & ((kept & 1) == 1))
        want = (kept + up).astype(np.uint16)
        assert np.array_equal(o.fwd(res, pre), want), (T, H)


def check_gr_fp64_emulation(o):
    rng = np.random.default_rng(58)
    g = random_bf16(rng, (3, 33), scale=3.0)
    pre = rng.random((3, 4), dtype=np.float32) * np.float32(5.0)
    prod = (pre.astype(np.float64)[:, :, None] * bf16_widen(g).astype(np.float64)[:, None, :]).astype(np.float32)
    bits = prod.view(np.uint32)
    kept = bits >> 16
    dropped = bits & 0xFFFF
    up = (dropped > 0x8000) | ((dropped == 0x8000) & ((kept & 1) == 1))
    assert np.array_equal(o.grad_residual(g, pre), (kept + up).astype(np.uint16))


ALL_CHECKS += [
    check_fwd_fp64_emulation,
    check_gr_fp64_emulation,
    check_f16_golden,
    check_f16_roundtrip_exhaustive,
    check_f16_vs_torch,
    check_agg_golden,
    check_agg_n4_bf16_is_the_pages_op,
    check_agg_exact_rational,
    check_agg_one_hot,
    check_agg_grad_residual_exact,
    check_agg_grad_pre_integer_exact,
    check_agg_grad_pre_order_f16,
]


# --------------------------------------------------------------------------
# the fused pre coefficients: pre = sigmoid(alpha * mix + b)
#
# Source: "perf: fuse mHC coefficient backward epilogue" (Liger-Kernel pull
# request 1402), Summary (pre / post sigmoid derivatives, grad_mix, grad_b and
# alpha gradients) and Risks and Limitations (deterministic order of the
# grad_b / alpha reductions).  The formulas are a reading; the binary32
# sigmoid is a definition of this library (exp32, sigmoid32 in the oracle).
# --------------------------------------------------------------------------

def f32_ulp(x) -> np.ndarray:
    """Spacing of binary32 at |x| (x given in FP64), never below the subnormal step."""
    a = np.abs(np.asarray(x, dtype=np.float64)).astype(np.float32)
    return np.maximum(np.spacing(a).astype(np.float64), 2.0 ** -149)


def dense_floats(lo_bits: int, hi_bits: int, step: int) -> np.ndarray:
    """Every step-th binary32 pattern in [lo_bits, hi_bits)."""
    return np.arange(lo_bits, hi_bits, step, dtype=np.uint64).astype(np.uint32).view(np.float32)


def sigmoid64(z) -> np.ndarray:
    """sigmoid in FP64 without overflow (accurate to a few FP64 ulps)."""
    z = np.asarray(z, dtype=np.float64)
    e = np.exp(-np.abs(z))
    return np.where(z >= 0, 1.0 / (1.0 + e), e / (1.0 + e))


def check_exp32_fp64_bound(o):
    """exp32 against FP64 e^x: within 1.2 binary32 ulps on [-104, 88.7] and
    correctly rounded on at least 99% of a dense sample (a dropped term, a
    one-part ln 2 or a wrong reduction breaks one of the two)."""
    neg = dense_floats(0x80000000, 0xC2D00000, 997)            # -0 .. -104
    pos = dense_floats(0x00000000, 0x42B17000, 1009)           # 0 .. 88.72
    edges = np.float32([-0.0, 0.0, -104.0, -87.33655, -0.34657359, -0.34657362,
                        -0.6931472, 0.6931472, 88.7, 88.72])
    x = np.concatenate([neg, pos, edges])
    y = o.exp32(x).astype(np.float64)
    ex = np.exp(x.astype(np.float64))
    err = np.abs(y - ex) / f32_ulp(ex)
    assert err.max() <= 1.2, f"max error {err.max():.3f} ulp at x={x[err.argmax()]}"
    exact = (y == ex.astype(np.float32).astype(np.float64)).mean()
    assert exact >= 0.99, f"only {exact:.4f} correctly rounded"


def _exp32_exact(x: float) -> float:
    """The defining step sequence of exp32, each binary32 operation done in
    exact rationals and rounded once (round_rne); x finite in [-104, 89]."""
    f32 = lambda v: round_rne(Fraction(v), 24)
    mul = lambda a, b: f32(Fraction(a) * Fraction(b))
    add = lambda a, b: f32(Fraction(a) + Fraction(b))
    log2e, l1, l2 = (float(f32_from_bits(u)) for u in (0x3FB8AA3B, 0x3F317200, 0x35BFBE8E))
    y = Fraction(mul(x, log2e))
    k = math.floor(y)
    if y - k > Fraction(1, 2) or (y - k == Fraction(1, 2) and k % 2 == 1):
        k += 1
    r = add(add(x, -mul(k, l1)), -mul(k, l2))
    c = [f32(Fraction(1, math.factorial(i))) for i in range(8)]
    q = c[7]
    for i in range(6, -1, -1):
        q = add(c[i], mul(r, q))
    k1 = int(k / 2)
    return f32(Fraction(f32(Fraction(q) * Fraction(2) ** k1)) * Fraction(2) ** (k - k1))


def check_exp32_exact_rational(o):
    """exp32 equals its step sequence done in exact rationals, including inputs
    where x * log2e rounds to exactly half an integer (the reduction's tie,
    broken to even) and results deep in the subnormal range."""
    log2e = f32_from_bits(0x3FB8AA3B)
    halves = np.arange(-149.5, 128.0, 1.0)
    x0 = (halves / np.float64(log2e)).astype(np.float32)
    cand = x0.view(np.int32)[:, None] + np.arange(-4, 5, dtype=np.int32)[None, :]
    cand = cand.astype(np.int32).view(np.float32)
    hit = (cand * log2e).astype(np.float32) == halves.astype(np.float32)[:, None]
    ties = cand[hit & (cand >= -104) & (cand <= 88.5)]
    assert ties.size > 100, f"only {ties.size} tie inputs found"
    rng = np.random.default_rng(90)
    xs = np.concatenate([np.float32(ties), np.float32([-103.9, -100.0, -88.0, -0.75, 3.0, 88.5]),
                         rng.uniform(-104, 88, 100).astype(np.float32)])
    got = o.exp32(xs)
    for x, g in zip(xs, got):
        assert float(g) == _exp32_exact(float(x)), f"x={x!r}: {g!r} vs {_exp32_exact(float(x))!r}"


def check_exp32_special(o):
    x = np.float32([0.0, -0.0, np.inf, -np.inf, np.nan, -104.5, 89.5, 1e30, -1e30])
    y = o.exp32(x)
    assert f32_bits(y[:2]).tolist() == [0x3F800000, 0x3F800000]
    assert y[2] == np.inf and f32_bits(y[3]) == 0 and np.isnan(y[4])
    assert f32_bits(y[5]) == 0 and y[6] == np.inf and y[7] == np.inf and f32_bits(y[8]) == 0


def check_sigmoid_golden(o):
    rows = list(golden_rows("sigmoid_worked_examples.txt"))
    z = np.array([f32_from_bits(int(r[1], 16)) for r in rows], dtype=np.float32)
    s, ds = o.sigmoid32(z)
    for (name, _, ws, wd), a, b in zip(rows, f32_bits(s), f32_bits(ds)):
        assert (int(a), int(b)) == (int(ws, 16), int(wd, 16)), f"{name}: {hex(a)} {hex(b)}"


def check_sigmoid_fp64_bound(o):
    """sigmoid within 2.5 ulps and sigmoid' within 4.5 ulps of FP64, for both
    signs of z on a dense sample of [-128, 128]."""
    zp = dense_floats(0x00000000, 0x43000000, 1013)
    z = np.concatenate([zp, -zp])
    s, ds = o.sigmoid32(z)
    S = sigmoid64(z)
    D = S * sigmoid64(-z.astype(np.float64))
    es = np.abs(s.astype(np.float64) - S) / f32_ulp(S)
    ed = np.abs(ds.astype(np.float64) - D) / f32_ulp(D)
    assert es.max() <= 2.5, f"sigmoid {es.max():.3f} ulp at z={z[es.argmax()]}"
    assert ed.max() <= 4.5, f"sigmoid' {ed.max():.3f} ulp at z={z[ed.argmax()]}"


def check_sigmoid_invariants(o):
    """sigmoid(z) + sigmoid(-z) is 1 within 2^-23 (the rounding of d = 1 + e
    moves (1 + e)/d off 1 by at most 2^-24, the two quotients add at most
    3 * 2^-26), sigmoid' is even (bit for bit), sigmoid is non-decreasing in z
    and lies in [0, 1]."""
    rng = np.random.default_rng(91)
    z = np.sort(np.concatenate([rng.standard_normal(20000).astype(np.float32) * np.float32(8.0),
                                dense_floats(0x3F000000, 0x41A00000, 40009)]))
    s, ds = o.sigmoid32(z)
    sn, dsn = o.sigmoid32(-z)
    assert np.all(np.abs(s.astype(np.float64) + sn.astype(np.float64) - 1.0) <= 2.0 ** -23)
    assert np.array_equal(f32_bits(ds), f32_bits(dsn))
    assert np.all(np.diff(s.astype(np.float64)) >= 0.0)
    assert np.all((s >= 0.0) & (s <= 1.0))


def _coeff_inputs(rng, T, n):
    mix = (rng.standard_normal((T, n)) * 2.0).astype(np.float32)
    alpha = np.float32(rng.uniform(0.2, 3.0))
    b = rng.standard_normal(n).astype(np.float32)
    return mix, alpha, b


def check_pre_sigmoid_wiring(o):
    """pre = sigmoid(RN(RN(alpha*mix) + b[k])) with the [T,n] layout (the
    pre-activation by numpy binary32 arithmetic), and within the FP64 bound of
    the exact sigmoid(alpha*mix + b)."""
    rng = np.random.default_rng(92)
    for n in (1, 2, 4, 8):
        T = 37
        mix, alpha, b = _coeff_inputs(rng, T, n)
        z = (alpha * mix).astype(np.float32) + b[None, :]
        want, _ = o.sigmoid32(z.astype(np.float32))
        got = o.pre_sigmoid(mix, alpha, b)
        assert np.array_equal(f32_bits(got), f32_bits(want)), n
        z64 = np.float64(alpha) * mix.astype(np.float64) + b.astype(np.float64)[None, :]
        S = sigmoid64(z64)
        dz = 2.02 * U * (np.abs(np.float64(alpha) * mix) + np.abs(b.astype(np.float64))[None, :])
        bound = 2.5 * f32_ulp(S) + S * (1.0 - S) * dz * 1.01
        assert np.all(np.abs(got.astype(np.float64) - S) <= bound), n


def check_agg_sigmoid_fwd_half(o):
    """mix = 0 and b = 0 give z = 0 and pre = 0.5 exactly, so the fused forward
    is the aggregate with pre = 0.5, emulated in exact rationals."""
    rng = np.random.default_rng(93)
    for dtype in ("bf16", "f16"):
        for n in (1, 2, 4, 8):
            T, H = 3, 19
            r = random_storage(rng, (T, n, H), dtype, scale=2.0)
            got = o.aggregate_sigmoid_fwd(r, np.zeros((T, n), np.float32), np.float32(1.7),
                                          np.zeros(n, np.float32), dtype)
            want = _agg_exact(r, np.full((T, n), 0.5, dtype=np.float32), dtype)
            assert np.array_equal(got, want), (dtype, n)


def check_agg_sigmoid_fwd_composition(o):
    rng = np.random.default_rng(94)
    for dtype, n, T, H in (("bf16", 4, 5, 33), ("f16", 8, 3, 17), ("bf16", 1, 4, 9)):
        r = random_storage(rng, (T, n, H), dtype)
        mix, alpha, b = _coeff_inputs(rng, T, n)
        got = o.aggregate_sigmoid_fwd(r, mix, alpha, b, dtype)
        assert np.array_equal(got, o.aggregate_fwd(r, o.pre_sigmoid(mix, alpha, b), dtype))


def check_agg_sigmoid_bwd_half(o):
    """z = 0: sigmoid' = 1/4 exactly, so with integer-valued g and r, grad_z is
    the exact integer sum / 4, grad_mix = RN(alpha * grad_z), and
    grad_residual = g / 2 exactly."""
    rng = np.random.default_rng(95)
    lut = np.array([bf16_bits_of(float(v)) for v in range(-8, 9)], dtype=np.uint16)
    half = np.array([bf16_bits_of(v / 2.0) for v in range(-8, 9)], dtype=np.uint16)
    for n in (1, 2, 4, 8):
        T, H = 3, 2053
        gi = rng.integers(-8, 9, size=(T, H))
        ri = rng.integers(-8, 9, size=(T, n, H))
        alpha = np.float32(1.3)
        gr, gz, gm = o.aggregate_sigmoid_bwd(lut[gi + 8], lut[ri + 8], np.zeros((T, n), np.float32),
                                             alpha, np.zeros(n, np.float32))
        exact = np.einsum("th,tkh->tk", gi, ri).astype(np.float64) / 4.0
        assert np.array_equal(gz.astype(np.float64), exact), n
        assert np.array_equal(f32_bits(gm), f32_bits(alpha * exact.astype(np.float32))), n
        assert np.array_equal(gr, np.broadcast_to(half[gi + 8][:, None, :], (T, n, H))), n


def check_agg_sigmoid_bwd_composition(o):
    """grad_residual and grad_pre are the plain backward's at pre = sigmoid(z);
    grad_z = RN(grad_pre * sigmoid'(z)); grad_mix = RN(alpha * grad_z)."""
    rng = np.random.default_rng(96)
    for dtype, n, T, H in (("bf16", 4, 4, 40), ("f16", 2, 3, 21), ("bf16", 8, 2, 16)):
        g = random_storage(rng, (T, H), dtype)
        r = random_storage(rng, (T, n, H), dtype)
        mix, alpha, b = _coeff_inputs(rng, T, n)
        gr, gz, gm = o.aggregate_sigmoid_bwd(g, r, mix, alpha, b, dtype)
        pre = o.pre_sigmoid(mix, alpha, b)
        gr2, gp = o.aggregate_bwd(g, r, pre, dtype)
        z = (alpha * mix).astype(np.float32) + b[None, :]
        _, ds = o.sigmoid32(z.astype(np.float32))
        assert np.array_equal(gr, gr2)
        assert np.array_equal(f32_bits(gz), f32_bits(gp * ds))
        assert np.array_equal(f32_bits(gm), f32_bits(alpha * gz))


def order256_reference(x) -> np.float32:
    """ORDER-256 over a sequence, written as an explicit expression tree and
    evaluated recursively in numpy binary32: chunk = adjacent-pair tree over 8
    values (+0 past the end), lane j = +0 then its chunks j, j+256, ... in
    increasing order, each group of 32 lanes and then the 8 groups folded by
    halving (element i with element i + half)."""
    x = np.asarray(x, dtype=np.float32)
    n_chunks = -(-len(x) // 8)

    def leaf(i):
        return x[i] if i < len(x) else np.float32(0.0)

    def adjacent_pairs(nodes):
        if len(nodes) == 1:
            return nodes[0]
        return adjacent_pairs([nodes[2 * i] + nodes[2 * i + 1] for i in range(len(nodes) // 2)])

    def halving(nodes):
        if len(nodes) == 1:
            return nodes[0]
        h = len(nodes) // 2
        return halving([nodes[i] + nodes[i + h] for i in range(h)])

    def lane(j, c):
        # value of lane j after all of its chunks below c
        if c < 0:
            return np.float32(0.0)
        return lane(j, c - 256) + adjacent_pairs([leaf(8 * c + e) for e in range(8)])

    def lane_value(j):
        last = j + 256 * ((n_chunks - 1 - j) // 256) if j < n_chunks else -1
        return lane(j, last)

    groups = [halving([lane_value(32 * w + i) for i in range(32)]) for w in range(8)]
    return halving(groups)


def check_param_grad_recursive_builder(o):
    """grad_b and grad_alpha equal the recursive ORDER-256 builder over tokens,
    bit for bit, on random data (T from 1 to past 2048 tokens, so that lanes
    hold several chunks and the last chunk is ragged)."""
    rng = np.random.default_rng(97)
    for T in (1, 5, 8, 13, 300, 2049, 2100):
        for n in (1, 4):
            gz = rng.standard_normal((T, n)).astype(np.float32)
            mix = rng.standard_normal((T, n)).astype(np.float32)
            gb, ga = o.sigmoid_param_grad(gz, mix)
            for k in range(n):
                assert f32_bits(gb[k]) == f32_bits(order256_reference(gz[:, k])), (T, n, k)
            prod = gz * mix
            per_token = prod[:, 0] if n == 1 else (prod[:, 0] + prod[:, 1]) + (prod[:, 2] + prod[:, 3])
            assert f32_bits(ga) == f32_bits(order256_reference(per_token)), (T, n)


def check_param_grad_integer_exact(o):
    rng = np.random.default_rng(98)
    for T in (1, 7, 8, 9, 2047, 2048, 2049, 4104):
        for n in (1, 2, 4, 8):
            gzi = rng.integers(-8, 9, size=(T, n))
            mi = rng.integers(-8, 9, size=(T, n))
            gb, ga = o.sigmoid_param_grad(gzi.astype(np.float32), mi.astype(np.float32))
            assert np.array_equal(gb.astype(np.float64), gzi.sum(axis=0).astype(np.float64)), (T, n)
            assert float(ga) == float((gzi * mi).sum()), (T, n)


def check_param_grad_order_golden(o):
    """The ORDER-256 golden cases with tokens in place of h: the listed values
    sit in column k of grad_z (mix = 1) and must give the listed grad_b[k]; at
    n = 1 the same cases give grad_alpha."""
    vals_of = {0x3F80: 1.0, 0x3380: 2.0 ** -24, 0x8000: -0.0}
    for name, H, k, _carrier, positions, expected in golden_rows("grad_pre_order_cases.txt"):
        T, k = int(H), int(k)
        col = np.zeros(T, dtype=np.float32)
        for item in positions.split(","):
            pos, v = item.split(":")
            if pos == "*":
                col[:] = vals_of[int(v, 16)]
            else:
                col[int(pos)] = vals_of[int(v, 16)]
        gz = np.zeros((T, 4), dtype=np.float32)
        gz[:, k] = col
        gb, _ = o.sigmoid_param_grad(gz, np.ones((T, 4), dtype=np.float32))
        want = np.zeros(4, dtype=np.uint32)
        want[k] = int(expected, 16)
        assert np.array_equal(f32_bits(gb), want), name
        _, ga = o.sigmoid_param_grad(col[:, None].copy(), np.ones((T, 1), dtype=np.float32))
        assert int(f32_bits(ga)) == int(expected, 16), name


def check_param_grad_fp64_bound(o):
    rng = np.random.default_rng(99)
    for T in (3, 1000, 4096):
        n = 4
        gz = rng.standard_normal((T, n)).astype(np.float32)
        mix = rng.standard_normal((T, n)).astype(np.float32)
        gb, ga = o.sigmoid_param_grad(gz, mix)
        g64 = gz.astype(np.float64)
        depth = order256_depth(T)
        for k in range(n):
            exact = math.fsum(g64[:, k])
            assert abs(float(gb[k]) - exact) <= 1.01 * depth * U * np.abs(g64[:, k]).sum(), (T, k)
        prod = g64 * mix.astype(np.float64)
        exact = math.fsum(prod.ravel())
        assert abs(float(ga) - exact) <= 1.01 * (depth + 3) * U * np.abs(prod).sum(), T


ALL_CHECKS += [
    check_exp32_fp64_bound,
    check_exp32_exact_rational,
    check_exp32_special,
    check_sigmoid_golden,
    check_sigmoid_fp64_bound,
    check_sigmoid_invariants,
    check_pre_sigmoid_wiring,
    check_agg_sigmoid_fwd_half,
    check_agg_sigmoid_fwd_composition,
    check_agg_sigmoid_bwd_half,
    check_agg_sigmoid_bwd_composition,
    check_param_grad_recursive_builder,
    check_param_grad_integer_exact,
    check_param_grad_order_golden,
    check_param_grad_fp64_bound,
]


# --------------------------------------------------------------------------
# mHC post (a reading; the pages name "MHC Post" but print no formula)
# --------------------------------------------------------------------------

def check_post_golden(o):
    for name, res_s, post_s, x_s, y_s, want in golden_rows("post_worked_examples.txt"):
        res_row = np.array([f32_from_bits(int(v, 16)) for v in res_s.split(",")], dtype=np.float32)
        n = len(res_row)
        res = np.zeros((1, n, n), dtype=np.float32)
        res[0, 0] = res_row
        res[0, 1:] = 0.5
        post = np.full((1, n), 0.25, dtype=np.float32)
        post[0, 0] = f32_from_bits(int(post_s, 16))
        x = np.array([[int(v, 16) for v in x_s.split(",")]], dtype=np.uint16).reshape(1, n, 1)
        y = np.array([[int(y_s, 16)]], dtype=np.uint16)
        got = o.post_fwd(x, y, post, res)
        assert int(got[0, 0, 0]) == int(want, 16), f"{name}: {hex(int(got[0, 0, 0]))}"


def _post_exact(x_u16, y_u16, post, res, dtype):
    widen, rnd, bits = STORAGE[dtype]
    x = widen(x_u16)
    y = widen(y_u16)
    T, n, H = x.shape
    out = np.empty((T, n, H), dtype=np.uint16)
    for t in range(T):
        for k in range(n):
            for h in range(H):
                p = [exact_mul(float(res[t, k, j]), float(x[t, j, h])) for j in range(n)]
                while len(p) > 1:
                    p = [exact_add(p[2 * i], p[2 * i + 1]) for i in range(len(p) // 2)]
                s = exact_add(p[0], exact_mul(float(post[t, k]), float(y[t, h])))
                out[t, k, h] = bits(rnd(s))
    return out


def check_post_exact_rational(o):
    rng = np.random.default_rng(301)
    for dtype in ("bf16", "f16"):
        for n in (1, 2, 4, 8):
            T, H = 2, 5
            x = random_storage(rng, (T, n, H), dtype, scale=2.0)
            y = random_storage(rng, (T, H), dtype, scale=2.0)
            post = rng.random((T, n), dtype=np.float32) * np.float32(2.0)
            res = rng.random((T, n, n), dtype=np.float32)
            assert np.array_equal(o.post_fwd(x, y, post, res, dtype), _post_exact(x, y, post, res, dtype)), (dtype, n)


def check_post_identity_and_zero(o):
    """res = I and post = 0 return x (numerically); x = 0 returns cvt(RN(post * y))."""
    rng = np.random.default_rng(302)
    for n in (1, 2, 4, 8):
        T, H = 3, 33
        x = random_bf16(rng, (T, n, H))
        y = random_bf16(rng, (T, H))
        res = np.broadcast_to(np.eye(n, dtype=np.float32), (T, n, n)).copy()
        out = o.post_fwd(x, y, np.zeros((T, n), np.float32), res)
        assert np.array_equal(bf16_widen(out), bf16_widen(x)), n
        post = rng.random((T, n), dtype=np.float32)
        out0 = o.post_fwd(np.zeros_like(x), y, post, rng.random((T, n, n), dtype=np.float32))
        want = (post[:, :, None] * bf16_widen(y)[:, None, :]).astype(np.float32)
        assert np.array_equal(bf16_widen(out0), bf16_widen(o.bf16_from_float(want))), n


def check_post_fp64_bound(o):
    rng = np.random.default_rng(303)
    T, H, n = 4, 300, 4
    x = random_bf16(rng, (T, n, H))
    y = random_bf16(rng, (T, H))
    post = rng.random((T, n), dtype=np.float32)
    res = rng.random((T, n, n), dtype=np.float32)
    terms = res.astype(np.float64)[:, :, :, None] * bf16_widen(x).astype(np.float64)[:, None, :, :]
    lift = post.astype(np.float64)[:, :, None] * bf16_widen(y).astype(np.float64)[:, None, :]
    exact = terms.sum(axis=2) + lift
    mag = np.abs(terms).sum(axis=2) + np.abs(lift)
    got = bf16_widen(o.post_fwd(x, y, post, res)).astype(np.float64)
    assert np.all(np.abs(got - exact) <= 0.5 * bf16_ulp(got) + 4.01 * U * mag)


def check_post_bwd_exact(o):
    """Integer-valued g, x, y: grad_res and grad_post are exact integer sums in any
    order; res = I gives grad_x = g and post = e_0 gives grad_y = g[:, 0]."""
    rng = np.random.default_rng(304)
    lut = np.array([bf16_bits_of(float(v)) for v in range(-8, 9)], dtype=np.uint16)
    for n in (1, 2, 4, 8):
        T, H = 2, 2053
        gi = rng.integers(-8, 9, size=(T, n, H))
        xi = rng.integers(-8, 9, size=(T, n, H))
        yi = rng.integers(-8, 9, size=(T, H))
        post = np.zeros((T, n), np.float32)
        post[:, 0] = 1.0
        res = np.broadcast_to(np.eye(n, dtype=np.float32), (T, n, n)).copy()
        gx, gy, gp, gr = o.post_bwd(lut[gi + 8], lut[xi + 8], lut[yi + 8], post, res)
        assert np.array_equal(gp.astype(np.float64), np.einsum("tkh,th->tk", gi, yi).astype(np.float64)), n
        assert np.array_equal(gr.astype(np.float64), np.einsum("tkh,tjh->tkj", gi, xi).astype(np.float64)), n
        assert np.array_equal(bf16_widen(gx), bf16_widen(lut[gi + 8])), n
        assert np.array_equal(bf16_widen(gy), bf16_widen(lut[gi[:, 0] + 8])), n


def check_post_bwd_tree_golden(o):
    """grad_x and grad_y take the mixing tree over k: the 'mix_tree_pairs' column
    [1+2^-8, 0, 2^-24, 2^-24] gives 0x3F81 (left to right would give 0x3F80)."""
    n, H = 4, 1
    col = np.array([f32_from_bits(0x3F808000), 0.0, 2.0 ** -24, 2.0 ** -24], dtype=np.float32)
    res = np.zeros((1, n, n), dtype=np.float32)
    res[0, :, 2] = col                        # column j = 2: res[k, 2] for k = 0..3
    post = col[None, :].copy()
    g = np.full((1, n, H), 0x3F80, dtype=np.uint16)
    x = np.full((1, n, H), 0x3F80, dtype=np.uint16)
    y = np.full((1, H), 0x3F80, dtype=np.uint16)
    gx, gy, _, _ = o.post_bwd(g, x, y, post, res)
    assert int(gx[0, 2, 0]) == 0x3F81 and int(gy[0, 0]) == 0x3F81, (hex(int(gx[0, 2, 0])), hex(int(gy[0, 0])))


def check_post_bwd_order_golden(o):
    """grad_post is summed in ORDER-256: the golden cases, with the values in
    row k of g and y = 1."""
    for name, H, k, carrier, positions, expected in golden_rows("grad_pre_order_cases.txt"):
        H, k = int(H), int(k)
        vals = np.zeros(H, dtype=np.uint16)
        for item in positions.split(","):
            pos, v = item.split(":")
            if pos == "*":
                vals[:] = int(v, 16)
            else:
                vals[int(pos)] = int(v, 16)
        n = 4
        g = np.zeros((1, n, H), dtype=np.uint16)
        g[0, k] = vals
        x = np.zeros((1, n, H), dtype=np.uint16)
        y = np.full((1, H), 0x3F80, dtype=np.uint16)
        _, _, gp, gr = o.post_bwd(g, x, y, np.ones((1, n), np.float32), np.ones((1, n, n), np.float32))
        assert int(f32_bits(gp)[0, k]) == int(expected, 16), name
        # the same sums for grad_res with x = 1 in row j = 3
        x[0, 3] = 0x3F80
        _, _, _, gr = o.post_bwd(g, x, y, np.ones((1, n), np.float32), np.ones((1, n, n), np.float32))
        assert int(f32_bits(gr)[0, k, 3]) == int(expected, 16), name


ALL_CHECKS += [
    check_post_golden,
    check_post_exact_rational,
    check_post_identity_and_zero,
    check_post_fp64_bound,
    check_post_bwd_exact,
    check_post_bwd_tree_golden,
    check_post_bwd_order_golden,
]


# ---------------------------------------------------------------------------
# mHC post with post = sigmoid(alpha * mix + b)
# ---------------------------------------------------------------------------

def check_post_sigmoid_fwd_half(o):
    """mix = 0 and b = 0 give z = 0 and post = 0.5 exactly: the forward is the
    post with post = 0.5, emulated in exact rationals."""
    rng = np.random.default_rng(310)
    for dtype in ("bf16", "f16"):
        for n in (1, 2, 4, 8):
            T, H = 2, 7
            x = random_storage(rng, (T, n, H), dtype, scale=2.0)
            y = random_storage(rng, (T, H), dtype, scale=2.0)
            res = rng.random((T, n, n), dtype=np.float32)
            got = o.post_sigmoid_fwd(x, y, np.zeros((T, n), np.float32), np.float32(1.7),
                                     np.zeros(n, np.float32), res, dtype)
            want = _post_exact(x, y, np.full((T, n), 0.5, dtype=np.float32), res, dtype)
            assert np.array_equal(got, want), (dtype, n)


def check_post_sigmoid_bwd_half(o):
    """z = 0: sigmoid' = 1/4 exactly, so with integer-valued g and y, grad_z is
    the exact integer sum of g*y / 4, grad_mix = RN(alpha * grad_z); with
    res = I, grad_x = g; grad_y = cvt(tree of g / 2) and grad_res the exact
    integer sums."""
    rng = np.random.default_rng(311)
    lut = np.array([bf16_bits_of(float(v)) for v in range(-8, 9)], dtype=np.uint16)
    for n in (1, 2, 4, 8):
        T, H = 2, 2053
        gi = rng.integers(-8, 9, size=(T, n, H))
        xi = rng.integers(-8, 9, size=(T, n, H))
        yi = rng.integers(-8, 9, size=(T, H))
        alpha = np.float32(1.3)
        res = np.broadcast_to(np.eye(n, dtype=np.float32), (T, n, n)).copy()
        gx, gy, gz, gm, gr = o.post_sigmoid_bwd(lut[gi + 8], lut[xi + 8], lut[yi + 8],
                                                np.zeros((T, n), np.float32), alpha,
                                                np.zeros(n, np.float32), res)
        exact = np.einsum("tkh,th->tk", gi, yi).astype(np.float64) / 4.0
        assert np.array_equal(gz.astype(np.float64), exact), n
        assert np.array_equal(f32_bits(gm), f32_bits(alpha * exact.astype(np.float32))), n
        assert np.array_equal(gr.astype(np.float64), np.einsum("tkh,tjh->tkj", gi, xi).astype(np.float64)), n
        assert np.array_equal(bf16_widen(gx), bf16_widen(lut[gi + 8])), n
        # grad_y = sum over k of g / 2: integers / 2, exact in BF16 while |sum| <= 256
        half_sum = gi.sum(axis=1).astype(np.float64) / 2.0
        assert np.array_equal(bf16_widen(gy).astype(np.float64), half_sum), n


def check_post_sigmoid_wiring(o):
    """Random mix, alpha, b: the forward and backward are post_fwd / post_bwd at
    post = sigmoid32(RN(RN(alpha * mix) + b[k])) (pre-activation by numpy
    binary32 arithmetic), grad_z = RN(grad_post * sigmoid'(z)) and
    grad_mix = RN(alpha * grad_z)."""
    rng = np.random.default_rng(312)
    for dtype, n, T, H in (("bf16", 4, 4, 40), ("f16", 2, 3, 21), ("bf16", 8, 2, 16), ("f16", 1, 5, 9)):
        g = random_storage(rng, (T, n, H), dtype)
        x = random_storage(rng, (T, n, H), dtype)
        y = random_storage(rng, (T, H), dtype)
        res = rng.random((T, n, n), dtype=np.float32)
        mix, alpha, b = _coeff_inputs(rng, T, n)
        z = ((alpha * mix).astype(np.float32) + b[None, :]).astype(np.float32)
        post, ds = o.sigmoid32(z)
        assert np.array_equal(o.post_sigmoid_fwd(x, y, mix, alpha, b, res, dtype),
                              o.post_fwd(x, y, post, res, dtype)), (dtype, n)
        gx, gy, gz, gm, gr = o.post_sigmoid_bwd(g, x, y, mix, alpha, b, res, dtype)
        wx, wy, wp, wr = o.post_bwd(g, x, y, post, res, dtype)
        assert np.array_equal(gx, wx) and np.array_equal(gy, wy) and np.array_equal(gr, wr), (dtype, n)
        assert np.array_equal(f32_bits(gz), f32_bits((wp * ds).astype(np.float32))), (dtype, n)
        assert np.array_equal(f32_bits(gm), f32_bits((alpha * gz).astype(np.float32))), (dtype, n)


ALL_CHECKS += [
    check_post_sigmoid_fwd_half,
    check_post_sigmoid_bwd_half,
    check_post_sigmoid_wiring,
]


# --------------------------------------------------------------------------
# ORDER-256 over h: the oracle's row sums against the recursive builder
# --------------------------------------------------------------------------

#: row lengths that give lanes no chunk, one chunk or several, with ragged tails
RECURSIVE_H = tuple(range(1, 17)) + (255, 2047, 2049, 4104, 9001)


def _widen(u16, dtype):
    return bf16_widen(u16) if dtype == "bf16" else f16_widen(u16)


def check_gp_recursive_builder(o):
    """grad_pre equals the recursive ORDER-256 builder evaluated on the exact
    products g[t,h]*r[t,k,h] (a product of two 8- or 11-bit significands is
    exact in binary32), bit for bit, on random BF16 and FP16 data.  The
    builder shares nothing with the oracle's loops, so a different tree shape
    (another lane count, fold order or chunk tree) fails here on random data."""
    rng = np.random.default_rng(2563)
    for dtype in ("bf16", "f16"):
        for H in RECURSIVE_H:
            n = 4
            g = random_storage(rng, (1, H), dtype)
            r = random_storage(rng, (1, n, H), dtype)
            pre = np.ones((1, n), np.float32)
            _, gp = o.aggregate_bwd(g, r, pre, dtype)
            sums = [gp]
            if dtype == "bf16":
                sums.append(o.grad_pre(g, r))       # the pages' op (n = 4, BF16)
            q = _widen(g, dtype)[0][None, :] * _widen(r, dtype)[0]
            for k in range(n):
                want = f32_bits(order256_reference(q[k]))
                for s in sums:
                    assert f32_bits(s[0, k]) == want, (dtype, H, k)


def check_post_bwd_recursive_builder(o):
    """The mHC post's grad_post[t,k] = sum_h g[t,k,h]*y[t,h] and grad_res[t,k,j]
    = sum_h g[t,k,h]*x[t,j,h] equal the recursive ORDER-256 builder on the
    exact products, bit for bit (n = 2, BF16 and FP16)."""
    rng = np.random.default_rng(2564)
    n = 2
    for dtype in ("bf16", "f16"):
        for H in RECURSIVE_H:
            g = random_storage(rng, (1, n, H), dtype)
            x = random_storage(rng, (1, n, H), dtype)
            y = random_storage(rng, (1, H), dtype)
            post = np.ones((1, n), np.float32)
            res = np.ones((1, n, n), np.float32)
            _, _, gp, gr = o.post_bwd(g, x, y, post, res, dtype)
            gw, xw, yw = _widen(g, dtype)[0], _widen(x, dtype)[0], _widen(y, dtype)[0]
            for k in range(n):
                assert f32_bits(gp[0, k]) == f32_bits(order256_reference(gw[k] * yw)), \
                    ("grad_post", dtype, H, k)
                for j in range(n):
                    assert f32_bits(gr[0, k, j]) == f32_bits(order256_reference(gw[k] * xw[j])), \
                        ("grad_res", dtype, H, k, j)


ALL_CHECKS += [
    check_gp_recursive_builder,
    check_post_bwd_recursive_builder,
]

"""Forward parity on the GPU: the sm_103a kernels against the CPU oracle, byte
for byte, through the C ABI (forward_accuracy and forward_invariance).

Source of the contract: "Add batch-invariant h_aggregate kernel" -- Summary
(formula, shapes), Batch invariance (fixed tree, one writer, RN FP32, BF16 at
the boundaries) and Correctness (100 repeat calls byte-identical; a full batch
equals per-token calls byte for byte).
"""

import numpy as np
import pytest
import torch

import oracle
import _pins
from _gpu import (DevBuf, assert_bytes_equal, expected_fwd_path, lib, run_fwd, sha,
                  stream_handle, u16, f32)
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.inputs import forward_inputs, workload

pytestmark = pytest.mark.gpu

VEC32, VEC16 = binding.MHC_PATH_VEC32, binding.MHC_PATH_VEC16
PAIR, ELEMENT = binding.MHC_PATH_PAIR, binding.MHC_PATH_ELEMENT
SHIFT16 = binding.MHC_PATH_SHIFT16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


def oracle_fwd(res, pre):
    return oracle.fwd(u16(res), f32(pre))


# --- workload fwd_t129_h4096: T=129, H=4096, seed 0

def test_t129_bit_exact_and_split_invariant():
    w = workload("fwd_t129_h4096")
    (T, H), = w.shapes
    res, pre = forward_inputs(T, H, w.recipe, w.seed)
    full = run_fwd(res, pre, expect_path=VEC32)
    assert_bytes_equal(full, oracle_fwd(res, pre), "T=129 vs oracle")
    # 129 one-token calls (a different launch shape) give the same bytes
    r_d, p_d = res.cuda(), pre.cuda()
    out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    for t in range(T):
        binding.mhc_h_aggregate_fwd(r_d[t:t + 1], p_d[t:t + 1], out[t:t + 1])
    torch.cuda.synchronize()
    assert_bytes_equal(u16(out), full, "129 one-token calls vs full batch")


def test_t129_repeat_100_calls_byte_identical():
    res, pre = forward_inputs(129, 4096, "normal", 0, device="cpu")
    r_d, p_d = res.cuda(), pre.cuda()
    out = torch.empty((129, 4096), dtype=torch.bfloat16, device="cuda")
    digests = set()
    for _ in range(100):
        out.fill_(0)
        binding.mhc_h_aggregate_fwd(r_d, p_d, out)
        digests.add(sha(out))
    assert len(digests) == 1


# --- workload fwd_ragged: odd H and ragged shapes (realigned 16-byte path), seed 1

@pytest.mark.parametrize("T,H", workload("fwd_ragged").shapes)
def test_ragged_bit_exact(T, H):
    w = workload("fwd_ragged")
    res, pre = forward_inputs(T, H, w.recipe, w.seed)
    want = oracle_fwd(res, pre)
    for offsets in ((0, 0, 0), (2, 4, 2), (6, 0, 14), (4, 8, 10)):
        got = run_fwd(res, pre, offsets=offsets)
        assert_bytes_equal(got, want, f"ragged T={T} H={H} offsets={offsets}")
    if H % 2:
        assert expected_fwd_path(H, (0, 0, 0)) == SHIFT16   # odd H: 16-byte, realigned


# --- workload fwd_decode: decode-sized shapes, seed 2

@pytest.mark.parametrize("T,H", workload("fwd_decode").shapes)
def test_decode_bit_exact(T, H):
    w = workload("fwd_decode")
    res, pre = forward_inputs(T, H, w.recipe, w.seed)
    got = run_fwd(res, pre, expect_path=VEC32)
    assert_bytes_equal(got, oracle_fwd(res, pre), f"decode T={T} H={H}")


# --- workload fwd_prefill: every shape in full, with repeats and splits, in test_configs_gpu.py


# --- hand-worked elements through every path

@pytest.mark.parametrize("H,offsets,path", [
    (16, (0, 0, 0), VEC32), (8, (0, 0, 0), VEC16), (16, (16, 0, 0), VEC16), (8, (4, 0, 4), PAIR),
    (9, (0, 0, 0), ELEMENT), (8, (2, 4, 0), ELEMENT), (67, (0, 0, 0), SHIFT16),
    (72, (2, 0, 4), SHIFT16), (80, (2, 4, 0), SHIFT16), (64, (14, 0, 6), SHIFT16)])
def test_worked_examples_on_gpu(H, offsets, path):
    cases = list(_pins._fwd_cases())
    T = len(cases)
    rng = np.random.default_rng(31)
    res = _pins.random_bf16(rng, (T, 4, H))
    pre = rng.random((T, 4), dtype=np.float32)
    want = []
    for t, (name, r, p, expected) in enumerate(cases):
        res[t, :, H // 2] = r
        pre[t] = p
        want.append(expected)
    res_t = torch.from_numpy(res.view(np.int16).copy()).view(torch.bfloat16)
    got = run_fwd(res_t, torch.from_numpy(pre), offsets=offsets, expect_path=path)
    assert [int(v) for v in got[:, H // 2]] == want
    assert_bytes_equal(got, oracle.fwd(res, pre), "worked-example batch")


# --- all paths give the same bytes

@pytest.mark.parametrize("T,H", [(37, 1024), (5, 8), (300, 7168), (1, 4104), (3, 2050)])
def test_paths_agree(T, H):
    res, pre = forward_inputs(T, H, "decode", 9)
    want = oracle_fwd(res, pre)
    seen = set()
    for offsets in ((0, 0, 0), (0, 4, 0), (16, 0, 0), (0, 0, 16), (4, 0, 0), (0, 0, 8),
                    (2, 0, 0), (0, 0, 6)):
        seen.add(expected_fwd_path(H, offsets))
        got = run_fwd(res, pre, offsets=offsets)
        assert_bytes_equal(got, want, f"T={T} H={H} offsets={offsets}")
    assert seen & {ELEMENT, SHIFT16}


# --- edge cases

@pytest.mark.parametrize("T,H", [(1, 1), (1, 2), (3, 1), (2, 7), (1, 8), (7, 9), (64, 16),
                                 (513, 8), (2, 2056), (1, 65536), (3, 100000)])
def test_small_and_odd_shapes(T, H):
    res, pre = forward_inputs(T, H, "ragged", 10)
    got = run_fwd(res, pre)
    assert_bytes_equal(got, oracle_fwd(res, pre), f"T={T} H={H}")


def test_zero_tokens_launches_nothing():
    o = DevBuf(64)
    assert binding.fwd_raw(0, 0, o.ptr, 0, 4096, stream_handle()) == binding.MHC_OK
    torch.cuda.synchronize()
    assert np.all(o.get(np.uint8) == 0xA5)


def test_special_values():
    """Infinities from overflow, subnormal results, signed zeros, all finite inputs."""
    T, H = 16, 64
    rng = np.random.default_rng(33)
    res = _pins.random_bf16(rng, (T, 4, H), scale=1e4)
    res[0] = 0x8000                                   # -0 rows
    res[1, :, ::3] = 0x0001                           # BF16 subnormals
    res[2, :, :] = 0x7F7F                             # largest finite BF16
    pre = rng.random((T, 4), dtype=np.float32)
    pre[2] = 3.0e38                                   # overflow to inf
    pre[3] = 0.0
    pre[4] = -0.0
    pre[5] = np.float32(1e-40)                        # subnormal pre
    res_t = torch.from_numpy(res.view(np.int16).copy()).view(torch.bfloat16)
    pre_t = torch.from_numpy(pre)
    for offsets in ((0, 0, 0), (16, 0, 16), (4, 0, 4), (2, 0, 2)):
        got = run_fwd(res_t, pre_t, offsets=offsets)
        assert_bytes_equal(got, oracle.fwd(res, pre), f"special values offsets={offsets}")


def test_non_default_stream_and_tensor_api():
    res, pre = forward_inputs(77, 2048, "normal", 12)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        r_d, p_d = res.cuda(), pre.cuda()
        out = binding.h_aggregate(r_d, p_d, stream=s)
    s.synchronize()
    assert_bytes_equal(u16(out), oracle_fwd(res, pre), "side stream")


def test_rejected_call_writes_nothing():
    res, pre = forward_inputs(4, 64, "normal", 13, device="cuda")
    before = res.clone()
    # an output that overlaps the residual is rejected before any launch
    st = binding.fwd_raw(res.data_ptr(), pre.data_ptr(), res.data_ptr() + 16, 4, 64,
                         stream_handle())
    assert st == binding.MHC_ERR_INVALID_ARG
    overlapping = res.view(-1)[8:8 + 4 * 64].view(4, 64)
    with pytest.raises(binding.MhcError):
        binding.mhc_h_aggregate_fwd(res, pre, overlapping)
    torch.cuda.synchronize()
    assert torch.equal(res.view(torch.int16), before.view(torch.int16))


# --- the page's third check: against a plain PyTorch computation within its tolerance

@pytest.mark.parametrize("T,H", [(1, 4096), (8, 4096), (128, 7168), (1024, 7168), (3, 1279)])
def test_matches_plain_pytorch_within_page_tolerance(T, H):
    """"Add batch-invariant h_aggregate kernel", Correctness, check 3: the
    result matches a PyTorch reference within atol=5e-2, rtol=1e-2.  The
    reference here is plain PyTorch in FP32 on the CPU, rounded to BF16 once."""
    res, pre = forward_inputs(T, H, "normal", 77)
    out = binding.h_aggregate(res.cuda(), pre.cuda()).cpu().float()
    r = res.float()
    ref = ((pre[:, 0:1] * r[:, 0] + pre[:, 1:2] * r[:, 1]) +
           (pre[:, 2:3] * r[:, 2] + pre[:, 3:4] * r[:, 3])).to(torch.bfloat16).float()
    assert torch.allclose(out, ref, atol=5e-2, rtol=1e-2)

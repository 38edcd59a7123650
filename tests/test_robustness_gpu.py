"""Robustness on the GPU: the split launch of very large calls, a seeded fuzz
over shapes / alignments / stream counts / storage types, CUDA-graph capture,
and concurrent calls from several host threads."""

import threading

import numpy as np
import pytest
import torch

import oracle
from _gpu import (DTYPE_NAME, assert_bytes_equal, lib, run_agg_bwd, run_agg_fwd, sha, u16, f32)
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.inputs import backward_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


def test_split_launch_beyond_2e31_vectors():
    """The vector forward indexes vectors with 32 bits and splits calls of
    2^31 vectors or more into launches over consecutive token ranges.  With
    n = 1, H = 16384 and the 16-byte path, T = 2^20 tokens make exactly 2^31
    vectors: the second launch holds the last token.  (34 GB residual + 34 GB
    out on the device.)  Checked for pre given and for pre computed from the
    mix."""
    T, H = 1 << 20, 16384
    dev = torch.device("cuda")
    buf_r = torch.empty(T * H + 8, dtype=torch.bfloat16, device=dev)
    buf_o = torch.empty(T * H + 8, dtype=torch.bfloat16, device=dev)
    res = buf_r[8:].view(T, 1, H)          # 16-byte but not 32-byte aligned -> 16-byte path
    out = buf_o[8:].view(T, H)
    gen = torch.Generator(device=dev).manual_seed(123)
    step = 1 << 28
    flat = res.view(-1)
    for i in range(0, T * H, step):
        flat[i:i + step] = torch.randn(min(step, T * H - i), generator=gen, device=dev).to(torch.bfloat16)
    pre = torch.rand((T, 1), generator=gen, device=dev)
    assert binding.agg_fwd_path_raw(res.data_ptr(), pre.data_ptr(), out.data_ptr(), T, 1, H) == \
        binding.MHC_PATH_VEC16
    binding.mhc_aggregate_fwd(res, pre, out)
    torch.cuda.synchronize()
    V = H // 8
    boundary = (2 ** 31 - 1) // V          # first token of the second launch
    for t in (0, 1, boundary - 1, boundary, T - 1):
        want = oracle.aggregate_fwd(u16(res[t:t + 1]), f32(pre[t:t + 1]), "bf16")
        assert_bytes_equal(u16(out[t:t + 1]), want, f"token {t}")
    # the same split with pre computed from the mix: the second launch's mix
    # rows start at the boundary token
    mix = torch.randn((T, 1), generator=gen, device=dev) * 3
    alpha = torch.full((1,), 1.25, device=dev)
    b = torch.full((1,), -0.5, device=dev)
    binding.mhc_aggregate_sigmoid_fwd(res, mix, alpha, b, out)
    torch.cuda.synchronize()
    for t in (0, 1, boundary - 1, boundary):
        want = oracle.aggregate_sigmoid_fwd(u16(res[t:t + 1]), f32(mix[t:t + 1]), np.float32(1.25),
                                            np.float32([-0.5]), "bf16")
        assert_bytes_equal(u16(out[t:t + 1]), want, f"sigmoid coefficients, token {t}")
    del buf_r, buf_o, res, out, flat
    torch.cuda.empty_cache()


def test_fuzz_shapes_alignments_streams_dtypes():
    rng = np.random.default_rng(2026)
    for case in range(60):
        n = int(rng.choice([1, 2, 4, 8]))
        dtype = torch.bfloat16 if rng.random() < 0.6 else torch.float16
        H = int(rng.choice([int(rng.integers(1, 300)), 8 * int(rng.integers(1, 1100)),
                            16 * int(rng.integers(1, 600))]))
        T = int(rng.integers(1, 40))
        g, res, pre = backward_inputs(T, H, str(rng.choice(["normal", "ragged", "decode"])),
                                      int(rng.integers(0, 10 ** 6)), n=n, dtype=dtype)
        offs = [int(rng.choice([0, 2, 4, 8, 16])) for _ in range(5)]
        offs[2] = int(rng.choice([0, 4, 8]))   # pre: 4-byte aligned
        offs[4] = int(rng.choice([0, 4, 8]))   # grad_pre: 4-byte aligned
        name = DTYPE_NAME[dtype]
        what = f"case {case}: n={n} {name} T={T} H={H} offsets={offs}"
        got = run_agg_fwd(res, pre, (offs[1], offs[2], offs[0]))
        assert_bytes_equal(got, oracle.aggregate_fwd(u16(res), f32(pre), name), "fwd " + what)
        gr, gp = run_agg_bwd(g, res, pre, tuple(offs))
        want_gr, want_gp = oracle.aggregate_bwd(u16(g), u16(res), f32(pre), name)
        assert_bytes_equal(gr, want_gr, "grad_residual " + what)
        assert_bytes_equal(gp, want_gp, "grad_pre " + what)


def test_cuda_graph_capture_and_replay():
    g, res, pre = backward_inputs(300, 7168, "normal", 11, device="cuda")
    out = torch.empty((300, 7168), dtype=torch.bfloat16, device="cuda")
    gr = torch.empty((300, 4, 7168), dtype=torch.bfloat16, device="cuda")
    gp = torch.empty((300, 4), dtype=torch.float32, device="cuda")
    binding.mhc_h_aggregate_fwd(res, pre, out)
    binding.mhc_h_aggregate_bwd(g, res, pre, gr, gp)
    torch.cuda.synchronize()
    ref = (sha(out), sha(gr), sha(gp))
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=s):
        binding.mhc_h_aggregate_fwd(res, pre, out)
        binding.mhc_h_aggregate_bwd(g, res, pre, gr, gp)
    for _ in range(3):
        out.zero_()
        gr.zero_()
        gp.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert (sha(out), sha(gr), sha(gp)) == ref


def test_concurrent_host_threads_on_separate_streams():
    jobs = []
    for i in range(6):
        n, dtype = [(4, torch.bfloat16), (8, torch.float16), (2, torch.bfloat16)][i % 3]
        g, res, pre = backward_inputs(64, 4096, "normal", 200 + i, n=n, dtype=dtype, device="cuda")
        jobs.append((g, res, pre))
    torch.cuda.synchronize()
    refs = []
    for g, res, pre in jobs:
        o = binding.aggregate(res, pre)
        a, b = binding.aggregate_backward(g, res, pre)
        torch.cuda.synchronize()
        refs.append((sha(o), sha(a), sha(b)))
    results = [None] * len(jobs)
    errors = []

    def worker(i):
        try:
            g, res, pre = jobs[i]
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for _ in range(20):
                    o = binding.aggregate(res, pre, stream=s)
                    a, b = binding.aggregate_backward(g, res, pre, stream=s)
            s.synchronize()
            results[i] = (sha(o), sha(a), sha(b))
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    assert results == refs

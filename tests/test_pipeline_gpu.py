"""HostPipeline: forward + backward over pinned host tensors in token chunks on
three streams gives the bytes of one device call (tokens are independent)."""

import pytest
import torch

from _gpu import lib, sha
from invariant_mhc_aggregate_gb300 import binding
from invariant_mhc_aggregate_gb300.inputs import backward_inputs
from invariant_mhc_aggregate_gb300.pipeline import HostPipeline

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return lib()


@pytest.mark.parametrize("T,H,n,dtype,chunk", [(1000, 7168, 4, torch.bfloat16, 128),
                                               (257, 4096, 8, torch.float16, 64),
                                               (5, 1279, 2, torch.bfloat16, 2)])
def test_pipeline_matches_device_call(T, H, n, dtype, chunk):
    g, res, pre = backward_inputs(T, H, "decode", 99, n=n, dtype=dtype)
    hg, hr, hp = g.pin_memory(), res.pin_memory(), pre.pin_memory()
    ho = torch.empty((T, H), dtype=dtype).pin_memory()
    hgr = torch.empty((T, n, H), dtype=dtype).pin_memory()
    hgp = torch.empty((T, n), dtype=torch.float32).pin_memory()
    d_out = binding.aggregate(res.cuda(), pre.cuda())
    d_gr, d_gp = binding.aggregate_backward(g.cuda(), res.cuda(), pre.cuda())
    torch.cuda.synchronize()
    for graphs in (True, False):
        pipe = HostPipeline(n, H, dtype, chunk_tokens=chunk, slots=3, graphs=graphs)
        # step 1 runs eagerly (and is captured), steps 2 and 3 replay the graph
        for _ in range(3):
            for t in (ho, hgr, hgp):
                t.zero_()
            pipe.step(hr, hp, hg, ho, hgr, hgp)
            pipe.synchronize()
            assert sha(ho) == sha(d_out) and sha(hgr) == sha(d_gr) and sha(hgp) == sha(d_gp)


def test_pipeline_replay_reads_new_host_values():
    """A replayed step copies the host tensors' current contents."""
    T, H, n = 300, 4096, 4
    g, res, pre = backward_inputs(T, H, "normal", 98)
    g2, res2, pre2 = backward_inputs(T, H, "ragged", 97)
    hg, hr, hp = g.pin_memory(), res.pin_memory(), pre.pin_memory()
    ho = torch.empty((T, H), dtype=torch.bfloat16).pin_memory()
    hgr = torch.empty((T, n, H), dtype=torch.bfloat16).pin_memory()
    hgp = torch.empty((T, n), dtype=torch.float32).pin_memory()
    pipe = HostPipeline(n, H, torch.bfloat16, chunk_tokens=128, slots=3)
    for _ in range(2):
        pipe.step(hr, hp, hg, ho, hgr, hgp)
    pipe.synchronize()
    hg.copy_(g2)
    hr.copy_(res2)
    hp.copy_(pre2)
    pipe.step(hr, hp, hg, ho, hgr, hgp)
    pipe.synchronize()
    d_out = binding.aggregate(res2.cuda(), pre2.cuda())
    d_gr, d_gp = binding.aggregate_backward(g2.cuda(), res2.cuda(), pre2.cuda())
    torch.cuda.synchronize()
    assert sha(ho) == sha(d_out) and sha(hgr) == sha(d_gr) and sha(hgp) == sha(d_gp)

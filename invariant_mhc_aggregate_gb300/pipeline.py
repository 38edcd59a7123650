"""Forward + backward over host-resident data, pipelined in token chunks.

For callers whose tensors live in (pinned) host memory.  Tokens are
independent and every output byte depends only on its own token (the
determinism contract of the C ABI), so the batch can be split into chunks of
tokens: while chunk i runs its two kernels, chunk i+1 is copied to the device
and chunk i-1 is copied back, on three CUDA streams.  The results are the same
bytes as one call over the whole batch.

Device memory is a fixed ring of `slots` chunk buffers, allocated once;
PyTorch provides the memory, streams and events, and every step of the
operation runs in the library's kernels (through ``binding``).

A step is launched from the host chunk by chunk (about a dozen calls each,
some 150 us of host time a chunk).  With ``graphs=True`` the first step on a
given set of host tensors runs eagerly and is then captured into a CUDA graph
that later steps on the same tensors replay (every copy and kernel still runs
each step): that removes the host time, which pays for small chunks, but
consecutive replays do not overlap one step's last copies back with the next
step's first copies in, so for large chunks eager steps are faster (measured
at T=4096, H=7168: 512 tokens eager 1.94 ms a step, as graphs 2.09 ms; 128
tokens eager 4.99 ms, as graphs 2.46 ms).  Eager steps are the default.

The default shape, 1024-token chunks in 5 slots, was the fastest eager one
measured at T=4096, H=7168 (median of 5 rounds of 30 steps): 1.83 ms a step,
95% of what the host link allows for the step's 587 MB of copies; 512 / 3
took 1.94 ms, 1024 / 3 2.14 ms, 1024 / 4 1.85 ms, 2048 / 3 1.84 ms, and one
4096-token chunk (no overlap within a step) 3.06 ms.
"""

from __future__ import annotations

import torch

from . import binding


class HostPipeline:
    """Runs forward + backward for host tensors of a fixed (n, H, dtype).

    step(residual, pre, g, out, grad_residual, grad_pre) reads residual
    [T,n,H], pre [T,n] and g [T,H] from host memory and writes out [T,H],
    grad_residual [T,n,H] and grad_pre [T,n] to host memory.  Host tensors
    should be pinned for the copies to overlap.  The call returns once the
    work is enqueued; ``synchronize()`` waits for it.
    """

    def __init__(self, n: int, H: int, dtype=torch.bfloat16, chunk_tokens: int = 1024,
                 slots: int = 5, device=None, graphs: bool = False):
        if dtype not in (torch.bfloat16, torch.float16):
            raise TypeError("dtype must be bfloat16 or float16")
        self.n, self.H, self.dtype = n, H, dtype
        self.chunk = int(chunk_tokens)
        self.device = torch.device(device) if device is not None else torch.device(
            "cuda", torch.cuda.current_device())
        C = self.chunk
        dev = self.device
        self.slots = []
        for _ in range(slots):
            self.slots.append(dict(
                res=torch.empty((C, n, H), dtype=dtype, device=dev),
                pre=torch.empty((C, n), dtype=torch.float32, device=dev),
                g=torch.empty((C, H), dtype=dtype, device=dev),
                out=torch.empty((C, H), dtype=dtype, device=dev),
                gr=torch.empty((C, n, H), dtype=dtype, device=dev),
                gp=torch.empty((C, n), dtype=torch.float32, device=dev),
                loaded=torch.cuda.Event(), computed=torch.cuda.Event(), drained=torch.cuda.Event(),
                used=False))
        self.h2d = torch.cuda.Stream(dev)
        self.compute = torch.cuda.Stream(dev)
        self.d2h = torch.cuda.Stream(dev)
        #: graph steps are captured from and replayed on this stream
        self.stream = torch.cuda.Stream(dev)
        self.graphs = bool(graphs)
        self._graphs = {}

    _MAX_GRAPHS = 8

    def step(self, residual, pre, g, out, grad_residual, grad_pre) -> None:
        args = (residual, pre, g, out, grad_residual, grad_pre)
        if not self.graphs:
            self._enqueue(args, fresh=False, join=False)
            return
        key = tuple((t.data_ptr(), tuple(t.shape), t.dtype) for t in args)
        graph = self._graphs.get(key)
        if graph is None:
            self._enqueue(args, fresh=False, join=True)    # this step's results
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=self.stream):
                self._enqueue(args, fresh=True, join=True)  # recorded for the next steps
            if len(self._graphs) >= self._MAX_GRAPHS:
                self._graphs.pop(next(iter(self._graphs)))
            self._graphs[key] = graph
            return
        with torch.cuda.stream(self.stream):
            graph.replay()

    def _enqueue(self, args, fresh: bool, join: bool) -> None:
        """The chunk loop.  `join`: fork the three streams from self.stream and
        join them back (graph capture and replay; eager steps skip it, so that
        one step's last copies back overlap the next step's first copies in).
        `fresh`: no earlier use of the slots to wait for."""
        residual, pre, g, out, grad_residual, grad_pre = args
        T = residual.shape[0]
        if join:
            for st in (self.h2d, self.compute, self.d2h):
                st.wait_stream(self.stream)
        if fresh:
            for s in self.slots:
                s["used"] = False
        for i, t0 in enumerate(range(0, T, self.chunk)):
            t1 = min(T, t0 + self.chunk)
            m = t1 - t0
            s = self.slots[i % len(self.slots)]
            with torch.cuda.stream(self.h2d):
                if s["used"]:
                    self.h2d.wait_event(s["drained"])       # the slot's last results are out
                s["res"][:m].copy_(residual[t0:t1], non_blocking=True)
                s["pre"][:m].copy_(pre[t0:t1], non_blocking=True)
                s["g"][:m].copy_(g[t0:t1], non_blocking=True)
                s["loaded"].record(self.h2d)
            with torch.cuda.stream(self.compute):
                self.compute.wait_event(s["loaded"])
                binding.mhc_aggregate_fwd(s["res"][:m], s["pre"][:m], s["out"][:m], self.compute)
                binding.mhc_aggregate_bwd(s["g"][:m], s["res"][:m], s["pre"][:m], s["gr"][:m],
                                          s["gp"][:m], self.compute)
                s["computed"].record(self.compute)
            with torch.cuda.stream(self.d2h):
                self.d2h.wait_event(s["computed"])
                out[t0:t1].copy_(s["out"][:m], non_blocking=True)
                grad_residual[t0:t1].copy_(s["gr"][:m], non_blocking=True)
                grad_pre[t0:t1].copy_(s["gp"][:m], non_blocking=True)
                s["drained"].record(self.d2h)
            s["used"] = True
        if join:
            for st in (self.h2d, self.compute, self.d2h):
                self.stream.wait_stream(st)

    def synchronize(self) -> None:
        self.stream.synchronize()
        self.d2h.synchronize()
        self.compute.synchronize()
        self.h2d.synchronize()

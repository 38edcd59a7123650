"""The multi-rank host logic on CPU with the gloo backend (world size 2).

The path shards over tokens with no exchange: each rank computes its own
contiguous token range, and the gathered results equal one call over the whole
batch byte for byte.  Only the benchmark's timing uses a collective (the
maximum of the per-rank step times).
"""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

from invariant_mhc_aggregate_gb300.sharding import token_range  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("T,world", [(0, 2), (1, 2), (7, 2), (8, 4), (129, 3), (4096, 8)])
def test_token_ranges_partition_the_batch(T, world):
    ranges = [token_range(T, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == T
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a1 == b0
    sizes = [b - a for a, b in ranges]
    assert max(sizes) - min(sizes) <= 1


def test_token_range_rejects_bad_requests():
    with pytest.raises(ValueError):
        token_range(10, 2, 2)
    with pytest.raises(ValueError):
        token_range(10, 0, 0)


def _worker(rank, world, port, T, H, out_path):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    import bench
    from invariant_mhc_aggregate_gb300.inputs import backward_inputs
    dist.init_process_group("gloo", rank=rank, world_size=world)
    g, res, pre = backward_inputs(T, H, "ragged", seed=21)       # the same global batch on every rank
    a, b = token_range(T, rank, world)
    u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    out = oracle.fwd(u16(res[a:b]), pre[a:b].numpy())
    gr, gp = oracle.bwd(u16(g[a:b]), u16(res[a:b]), pre[a:b].numpy())
    parts = [None] * world
    dist.all_gather_object(parts, (a, b, out.tobytes(), gr.tobytes(), gp.tobytes()))
    step_max = bench.max_over_ranks(1.0 + rank, dist, "cpu")
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump({"parts": [(p[0], p[1], p[2].hex(), p[3].hex(), p[4].hex()) for p in parts],
                       "step_max": step_max}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_match_one_call(tmp_path):
    import oracle
    from invariant_mhc_aggregate_gb300.inputs import backward_inputs
    T, H, world = 13, 1279, 2
    out_path = str(tmp_path / "gathered.json")
    mp.start_processes(_worker, args=(world, _free_port(), T, H, out_path), nprocs=world,
                       start_method="spawn", join=True)
    got = json.load(open(out_path))
    assert got["step_max"] == 2.0
    g, res, pre = backward_inputs(T, H, "ragged", seed=21)
    u16 = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    full_out = oracle.fwd(u16(res), pre.numpy())
    full_gr, full_gp = oracle.bwd(u16(g), u16(res), pre.numpy())
    cat = lambda i: b"".join(bytes.fromhex(p[i]) for p in got["parts"])
    assert [tuple(p[:2]) for p in got["parts"]] == [token_range(T, r, world) for r in range(world)]
    assert cat(2) == full_out.tobytes()
    assert cat(3) == full_gr.tobytes()
    assert cat(4) == full_gp.tobytes()


def test_torchrun_reference_arm_prints_one_line():
    """`bench.py --impl reference` under a 2-rank launch: rank 0 runs the CPU
    oracle and prints one JSON line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "0", "--T", "256", "--H", "1024"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0

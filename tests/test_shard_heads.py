"""The head partition of one problem across ranks (``head_range``,
``sdpa_forward_heads``, ``bench.py --shard heads``).  Every (batch, head) of
the forward is independent, so ranks that each compute their contiguous
range of heads produce the whole output between them with no exchange.  On
the CPU: the split's coverage, and gloo ranks that each compute their range
with the fp64 oracle and gather it; on the GPU: per-range calls reproduce the
whole call bit for bit."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
import sdpa_inputs
from scaled_dot_product_forward_gb300 import head_range


@pytest.mark.parametrize("world", [1, 2, 3, 4, 7, 8, 32])
@pytest.mark.parametrize("n_heads", [1, 4, 16, 32, 33, 128])
def test_head_ranges_cover_every_head_once(n_heads, world):
    ranges = [head_range(n_heads, r, world) for r in range(world)]
    assert ranges[0][0] == 0 and ranges[-1][1] == n_heads
    assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
    sizes = [h1 - h0 for h0, h1 in ranges]
    assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 0


def test_head_range_rejects_bad_ranks():
    for args in [(8, 2, 2), (8, -1, 2), (8, 0, 0), (-1, 0, 1)]:
        with pytest.raises(ValueError):
            head_range(*args)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    qq, kk, vv = sdpa_inputs.custom((2, 5, 40, 16), dtype=torch.bfloat16, seed=1500)[:3]
    h0, h1 = head_range(5, rank, world)
    part = torch.from_numpy(oracle.sdpa(qq[:, h0:h1], kk[:, h0:h1], vv[:, h0:h1],
                                        is_causal=True))
    # gather the ranges (padded to the largest) on every rank
    size = torch.tensor([h1 - h0])
    sizes = [torch.zeros_like(size) for _ in range(world)]
    dist.all_gather(sizes, size)
    hmax = int(max(s.item() for s in sizes))
    pad = torch.zeros(2, hmax, 40, 16, dtype=torch.float64)
    pad[:, :h1 - h0] = part
    parts = [torch.zeros_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad)
    whole = torch.cat([p[:, :int(s.item())] for p, s in zip(parts, sizes)], dim=1)
    q.put((rank, whole.numpy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_together_give_the_whole_output(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    qq, kk, vv = sdpa_inputs.custom((2, 5, 40, 16), dtype=torch.bfloat16, seed=1500)[:3]
    ref = oracle.sdpa(qq, kk, vv, is_causal=True)
    for r in range(world):
        assert np.array_equal(got[r], ref)


@pytest.mark.gpu
@pytest.mark.parametrize("world", [2, 3, 5])
def test_head_ranges_reproduce_the_whole_call(sdpa_lib, world):
    """Each rank's range computed in turn on one GPU into one output buffer:
    bit-identical to one call over all heads (per-head arithmetic does not
    depend on which heads share the launch)."""
    qh, kh, vh = sdpa_inputs.custom((2, 16, 640, 128), dtype=torch.bfloat16, seed=1510)[:3]
    qd, kd, vd = (x.cuda() for x in (qh, kh, vh))
    whole = sdpa_lib.sdpa_forward(qd, kd, vd, is_causal=True)
    out = torch.full_like(qd, float("nan"))
    for r in range(world):
        sdpa_lib.sdpa_forward_heads(qd, kd, vd, out, *head_range(16, r, world), is_causal=True)
    torch.cuda.synchronize()
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    assert torch.equal(out, whole)


def test_job_rate_counts_the_work_once_when_sharded():
    import bench
    from scaled_dot_product_forward_gb300 import head_range
    total = 5.5e11
    # heads split over 3 ranks: each did its share, the job did the workload once
    shares = [total * (h1 - h0) / 32 for h0, h1 in (head_range(32, r, 3) for r in range(3))]
    assert abs(sum(shares) - total) < 1.0
    assert bench.job_flops(total, shares[0], 3, sharded=True) == total
    # replicas: every rank ran the whole workload
    assert bench.job_flops(total, total, 4, sharded=False) == 4 * total
    assert bench.job_flops(total, total, 1, sharded=True) == total

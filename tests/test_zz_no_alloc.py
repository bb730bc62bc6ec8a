"""The masked forward that allocates nothing (sdpa_forward_masked_noalloc).

Some callers cannot allocate device memory: code running inside another
runtime whose memory pool already holds the device's memory, or a serving
loop that must not call cudaMalloc / cudaFree because they can synchronise
the whole device.  For them the mask summary sits in one fixed array inside
the library (enough for L <= 4096).  Several calls in a row -- different
masks, sizes, ranks and head sizes, the first filling the whole array at
L = 4096, so each later call reads an array the previous one left behind --
must agree with sdpa_forward and with the fp64 oracle within the parity
tolerance, fully removed rows must be exactly zero, a call must not change
the device's free memory, and a mask larger than the array's limit is
refused.  This file is collected last; it passes alone and after the other
tests."""
import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from tests.test_parity import check

pytestmark = pytest.mark.gpu

SDPA_ERR_SHAPE = 3
MAX_L = 4096


def cases():
    i = torch.arange(640)
    return [
        # (shape, dtype, mask): L = 4096 uses the whole fixed array
        ((1, 2, 4096, 64), torch.float16,
         sdpa_inputs.bernoulli_mask(4096, 0.3, seed=73, n_full_rows=16, rows_seed=74)),
        ((1, 4, 1024, 64), torch.float16,
         sdpa_inputs.bernoulli_mask(1024, 0.3, seed=71, n_full_rows=4, rows_seed=72)),
        # rank 3 with a ragged L: the per-byte summary path (L % 16 != 0)
        ((3, 300, 64), torch.float16,
         sdpa_inputs.bernoulli_mask(300, 0.3, seed=75, n_full_rows=3, rows_seed=76)),
        ((2, 2, 640, 128), torch.bfloat16,
         ((i[:, None] - i[None, :]).abs() >= 150).to(torch.uint8)),
    ]


def test_calls_in_a_row_match_sdpa_forward_and_the_oracle(sdpa_lib):
    for shape, dtype, mask in cases():
        q, k, v = sdpa_inputs.custom(shape, dtype=dtype, seed=shape[-2])
        qd, kd, vd, md = (x.cuda() for x in (q, k, v, mask))
        out = torch.full_like(qd, float("nan"))
        assert sdpa_lib.sdpa_forward_masked_noalloc(qd, kd, vd, md, out) == 0
        ref_gpu = sdpa_lib.sdpa_forward(qd, kd, vd, mask=md)
        torch.cuda.synchronize()
        rc, detail = sdpa_lib.sdpa_last_device_status()
        assert rc == 0, f"device status {rc} bits {detail:#x}"
        got = out.double().cpu().numpy()
        check(got, ref_gpu.double().cpu().numpy(), f"no-alloc vs sdpa_forward {shape}")
        check(got, oracle.sdpa(q, k, v, mask=mask), f"no-alloc vs oracle {shape}")
        dead = torch.nonzero(mask.bool().all(dim=1)).flatten().numpy()
        assert np.all(got[..., dead, :] == 0.0)


def test_a_call_allocates_no_device_memory(sdpa_lib):
    shape, dtype, mask = cases()[1]
    q, k, v = (x.cuda() for x in sdpa_inputs.custom(shape, dtype=dtype, seed=5))
    md = mask.cuda()
    out = torch.empty_like(q)
    stream = torch.cuda.Stream()
    assert sdpa_lib.sdpa_forward_masked_noalloc(q, k, v, md, out, stream=stream) == 0  # warm-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert sdpa_lib.sdpa_forward_masked_noalloc(q, k, v, md, out, stream=stream) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert sdpa_lib.sdpa_last_device_status()[0] == 0


def test_mask_beyond_the_array_is_refused(sdpa_lib):
    L = MAX_L + 1
    q, k, v = (torch.zeros((1, 1, L, 64), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    out = torch.empty_like(q)
    mask = torch.zeros((L, L), dtype=torch.uint8, device="cuda")
    assert sdpa_lib.sdpa_forward_masked_noalloc(q, k, v, mask, out) == SDPA_ERR_SHAPE

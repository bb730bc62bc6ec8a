"""The masked forward that allocates nothing (sdpa_forward_masked_noalloc).

For callers that cannot allocate device memory -- another runtime's pool
already holds the device's memory, or a loop must not call cudaMalloc /
cudaFree because they can synchronise the device -- the mask summary sits in
one fixed array inside the library.  Two calls in a row (different masks,
sizes and head sizes, so the second rewrites what the first left in the
shared array) must agree with sdpa_forward within the parity tolerance, and
a mask larger than the array's limit is refused.  This file is collected
last; it passes alone and after the other tests."""
import ctypes
import math

import pytest
import torch

import sdpa_inputs
from tests.test_parity import check

pytestmark = pytest.mark.gpu

SDPA_ERR_SHAPE = 3
MAX_L = 4096


def noalloc(sdpa, q, k, v, out, mask):
    lib = sdpa.load_library()
    fn = lib.sdpa_forward_masked_noalloc
    i64p, vp = ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p
    fn.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, i64p, i64p, i64p, i64p, i64p,
                   vp, ctypes.c_float, vp]
    fn.restype = ctypes.c_int
    arr = lambda vals: (ctypes.c_int64 * len(vals))(*vals)
    dtype = 0 if q.dtype == torch.bfloat16 else 1
    st = torch.cuda.current_stream().cuda_stream
    return fn(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(out.data_ptr()), dtype,
              q.dim(), arr(q.shape), arr(q.stride()), arr(k.stride()), arr(v.stride()),
              arr(out.stride()), vp(mask.data_ptr()), ctypes.c_float(math.nan),
              vp(st) if st else None)


def test_two_calls_match_sdpa_forward(sdpa_lib):
    i = torch.arange(640)
    cases = [
        ((1, 4, 1024, 64), torch.float16,
         sdpa_inputs.bernoulli_mask(1024, 0.3, seed=71, n_full_rows=4, rows_seed=72)),
        ((2, 2, 640, 128), torch.bfloat16, ((i[:, None] - i[None, :]).abs() >= 150).to(torch.uint8)),
    ]
    for shape, dtype, mask in cases:
        q, k, v = (x.cuda() for x in sdpa_inputs.custom(shape, dtype=dtype, seed=shape[2]))
        md = mask.cuda()
        out = torch.full_like(q, float("nan"))
        assert noalloc(sdpa_lib, q, k, v, out, md) == 0
        ref = sdpa_lib.sdpa_forward(q, k, v, mask=md)
        torch.cuda.synchronize()
        rc, detail = sdpa_lib.sdpa_last_device_status()
        assert rc == 0, f"device status {rc} bits {detail:#x}"
        check(out.double().cpu().numpy(), ref.double().cpu().numpy(), f"no-alloc {shape}")


def test_mask_beyond_the_array_is_refused(sdpa_lib):
    L = MAX_L + 1
    q, k, v = (torch.zeros((1, 1, L, 64), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    out = torch.empty_like(q)
    mask = torch.zeros((L, L), dtype=torch.uint8, device="cuda")
    assert noalloc(sdpa_lib, q, k, v, out, mask) == SDPA_ERR_SHAPE

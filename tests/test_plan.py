"""Plans: validate and encode once, launch many times (sdpa_plan_*)."""
import ctypes

import pytest
import torch

import oracle
import sdpa_inputs
from tests.test_api import K, M, O, Q, V, contiguous
from scaled_dot_product_forward_gb300 import _build


@pytest.fixture(scope="module")
def lib():
    _build.build()
    import scaled_dot_product_forward_gb300 as sdpa
    return sdpa


def create(lib, q=Q, o=O, shape=(2, 3, 256, 64), causal=1, mask=None, rank=4, dtype=0):
    st = contiguous(shape)
    h = ctypes.c_void_p(None)
    arr = lambda vals: (ctypes.c_int64 * len(vals))(*vals)
    rc = lib.load_library().sdpa_plan_create(
        ctypes.byref(h), ctypes.c_void_p(q), ctypes.c_void_p(K), ctypes.c_void_p(V),
        ctypes.c_void_p(o), dtype, rank, arr(shape), arr(st), arr(st), arr(st), arr(st), causal,
        ctypes.c_void_p(mask) if mask else None, ctypes.c_float(float("nan")))
    return rc, h


def test_plan_create_validates_like_forward(lib):
    """Same argument checks and codes as sdpa_forward, before any CUDA call."""
    assert create(lib, q=0)[0] == 1
    assert create(lib, rank=5, shape=(1, 2, 3, 256, 64))[0] == 2
    assert create(lib, dtype=3)[0] == 4
    assert create(lib, shape=(2, 3, 256, 96))[0] == 3
    assert create(lib, q=Q + 8)[0] == 5
    assert create(lib, causal=1, mask=M)[0] == 6
    rc, h = create(lib, o=Q + 512)
    assert rc == 6 and not h.value
    c = lib.load_library()
    assert c.sdpa_plan_create(None, None, None, None, None, 0, 4, None, None, None, None,
                              None, 1, None, ctypes.c_float(1.0)) == 1
    assert c.sdpa_plan_launch(None, None) == 1
    assert c.sdpa_plan_set_pointers(None, None, None, None, None, None) == 1
    c.sdpa_plan_destroy(None)


@pytest.mark.gpu
def test_plan_matches_forward_and_rebinds(sdpa_lib):
    q, k, v = (x.cuda() for x in sdpa_inputs.custom((2, 3, 300, 128), seed=31))
    ref = sdpa_lib.sdpa_forward(q, k, v, is_causal=True)
    out = torch.empty_like(q)
    plan = sdpa_lib.SdpaPlan(q, k, v, out, is_causal=True)
    plan.launch()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    # rebind to other tensors of the same layout
    q2, k2, v2 = sdpa_inputs.custom((2, 3, 300, 128), seed=32)
    out2 = torch.empty_like(q)
    plan.set_pointers(q2.cuda(), k2.cuda(), v2.cuda(), out2)
    plan.launch()
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    got = out2.double().cpu().numpy()
    exp = oracle.sdpa(q2, k2, v2, is_causal=True)
    import numpy as np
    assert np.linalg.norm(got - exp) / np.linalg.norm(exp) <= 1e-2
    plan.close()


@pytest.mark.gpu
def test_plan_in_cuda_graph(sdpa_lib):
    """The launch is capturable: a graph of the plan replays the same result."""
    q, k, v, mask = sdpa_inputs.make(4)
    q, k, v, mask = q[:, :2].cuda(), k[:, :2].cuda(), v[:, :2].cuda(), mask.cuda()
    out = torch.empty_like(q)
    plan = sdpa_lib.SdpaPlan(q, k, v, out, mask=mask)
    s = torch.cuda.Stream()
    plan.launch(s)  # warm the launch path outside capture
    s.synchronize()
    ref = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.launch(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    plan.close()

"""Failure detection without a GPU fault: every barrier wait in the kernel is
bounded in time.  The test hook withholds the query-tile load, so the MMA and
softmax roles wait on a phase that never completes; each wait gives up after
the (shortened) limit, the CTA drains what it issued, frees its tensor memory
and records a status bit.  The host then reads SDPA_ERR_DEVICE_TIMEOUT and the
context stays usable: the next normal call is correct."""
import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [128, 64])
def test_withheld_load_times_out_and_recovers(sdpa_lib, D):
    q, k, v = sdpa_inputs.custom((1, 1, 256, D), seed=21)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    try:
        sdpa_lib.sdpa_debug_set_wait_limit_ns(50_000_000)  # 50 ms per wait
        sdpa_lib.sdpa_debug_withhold_q_load(True)
        sdpa_lib.sdpa_forward(qd, kd, vd, is_causal=True)
        rc, detail = sdpa_lib.sdpa_last_device_status()
    finally:
        sdpa_lib.sdpa_debug_withhold_q_load(False)
        sdpa_lib.sdpa_debug_set_wait_limit_ns(0)
    assert rc == 8, f"expected SDPA_ERR_DEVICE_TIMEOUT, got {rc}"
    assert detail & 1
    assert detail & ((1 << 1) | (1 << 4)), f"expected a Q or S wait site, bits {detail:#x}"
    # the status word was cleared and the context still works
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    out = sdpa_lib.sdpa_forward(qd, kd, vd, is_causal=True)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    ref = oracle.sdpa(q, k, v, is_causal=True)
    got = out.double().cpu().numpy()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-2
    assert torch.cuda.synchronize() is None


def test_sparse_withheld_load_times_out_and_recovers(sdpa_lib):
    """The same for the sparse top-k kernel: with Q withheld no product is
    ever issued, the gathers fill the ring and give up on a free stage, the
    softmax gives up on S; the next call is correct."""
    total_q, total_k, H, D, topk = 6, 600, 64, 128, 300
    q = sdpa_inputs.custom((total_q, H, D), seed=31)[0]
    kv = sdpa_inputs.custom((total_k, 1, D), seed=32)[0][:, 0].contiguous()
    rng = np.random.default_rng(33)
    idx = np.stack([rng.choice(total_k, topk, replace=False) for _ in range(total_q)]).astype(np.int32)
    qd, kvd, idd = q.cuda(), kv.cuda(), torch.from_numpy(idx).cuda()
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    try:
        sdpa_lib.sdpa_debug_set_wait_limit_ns(50_000_000)  # 50 ms per wait
        sdpa_lib.sdpa_debug_withhold_q_load(True)
        sdpa_lib.sdpa_sparse_forward(qd, kvd, kvd, idd)
        rc, detail = sdpa_lib.sdpa_last_device_status()
    finally:
        sdpa_lib.sdpa_debug_withhold_q_load(False)
        sdpa_lib.sdpa_debug_set_wait_limit_ns(0)
    assert rc == 8, f"expected SDPA_ERR_DEVICE_TIMEOUT, got {rc}"
    assert detail & 1
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    out = sdpa_lib.sdpa_sparse_forward(qd, kvd, kvd, idd)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    ref = oracle.sdpa_sparse(q, kv, kv, idx)
    got = out.double().cpu().numpy()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-2

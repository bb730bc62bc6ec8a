"""GPU parity of the log-sum-exp output (sdpa_forward_lse / plan.set_lse)
against the fp64 oracle.  The LSE is computed in fp32 from the running max
and sum of the online softmax, so the bound is absolute 2e-3 (the scores are
O(10)); rows with no admissible key must be exactly -inf, and the attention
output itself must be identical to a call without the LSE."""
import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs

pytestmark = pytest.mark.gpu
LSE_ATOL = 2e-3


def check_lse(got, ref):
    got = np.asarray(got, dtype=np.float64)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin)
    assert np.all(got[~fin] == -np.inf)
    err = np.abs(got[fin] - ref[fin]).max() if fin.any() else 0.0
    assert err <= LSE_ATOL, err


@pytest.mark.parametrize("shape,causal,dtype", [
    ((1, 2, 300, 128), True, torch.bfloat16),
    ((2, 1, 129, 64), False, torch.float16),
    ((3, 200, 64), True, torch.bfloat16),
])
def test_lse_small(sdpa_lib, shape, causal, dtype):
    q, k, v = sdpa_inputs.custom(shape, dtype=dtype, seed=60 + shape[-2])
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    out, lse = sdpa_lib.sdpa_forward(qd, kd, vd, is_causal=causal, return_lse=True)
    plain = sdpa_lib.sdpa_forward(qd, kd, vd, is_causal=causal)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    assert torch.equal(out, plain)
    _, ref = oracle.sdpa(q, k, v, is_causal=causal, return_lse=True)
    assert tuple(lse.shape) == tuple(shape[:-1])
    check_lse(lse.cpu().numpy(), ref)


def test_lse_masked_empty_rows(sdpa_lib):
    L = 256
    q, k, v = sdpa_inputs.custom((1, 2, L, 64), dtype=torch.float16, seed=70)
    mask = sdpa_inputs.bernoulli_mask(L, 0.3, seed=71, n_full_rows=6, rows_seed=72)
    out, lse = sdpa_lib.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), mask=mask.cuda(),
                                     return_lse=True)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    _, ref = oracle.sdpa(q, k, v, mask=mask, return_lse=True)
    assert np.isinf(ref).sum() == 2 * 6
    check_lse(lse.cpu().numpy(), ref)


def test_lse_strided_buffer_and_plan(sdpa_lib):
    """An LSE view with non-unit strides, through a plan."""
    q, k, v = (x.cuda() for x in sdpa_inputs.custom((2, 3, 200, 64), seed=80))
    out = torch.empty_like(q)
    big = torch.full((2, 200, 3), float("nan"), dtype=torch.float32, device="cuda")
    lse = big.permute(0, 2, 1)  # [B, H, L] view, strides (600, 1, 3)
    plan = sdpa_lib.SdpaPlan(q, k, v, out, is_causal=True)
    plan.set_lse(lse)
    plan.launch()
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    _, ref = oracle.sdpa(q.cpu(), k.cpu(), v.cpu(), is_causal=True, return_lse=True)
    check_lse(lse.cpu().numpy(), ref)
    plan.close()


def test_lse_headline_workload_sampled(sdpa_lib):
    w = sdpa_inputs.WORKLOADS[3]
    q, k, v, _ = sdpa_inputs.make(w)
    out, lse = sdpa_lib.sdpa_forward(q.cuda(), k.cuda(), v.cuda(), is_causal=True,
                                     return_lse=True)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    rows = sdpa_inputs.sample_rows(w.B, w.H, w.L, 128, seed=33)
    _, ref = oracle.sdpa_rows(q, k, v, rows.numpy(), is_causal=True, return_lse=True)
    got = lse.cpu()[rows[:, 0], rows[:, 1], rows[:, 2]].numpy()
    check_lse(got, ref)

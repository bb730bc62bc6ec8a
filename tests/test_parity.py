"""GPU parity: the sm_103a kernel, called through the C ABI, against the fp64
oracle on the same seeded inputs.

Tolerance (bf16/fp16 inputs, fp32 accumulation): L2-relative error <= 1e-2
and max-abs error <= 2e-2 over every compared element.  Rows with no
admissible key must be exactly zero.  Small and medium cases are compared
in full here; the five specified workloads at full size are compared in full
in test_parity_full.py, and a 131072-long sequence on sampled rows below.
"""
import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs

pytestmark = pytest.mark.gpu

L2_TOL, MAX_TOL = 1e-2, 2e-2


def check(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = got - ref
    nref = np.linalg.norm(ref)
    l2 = np.linalg.norm(err) / (nref if nref > 0 else 1.0)
    mx = np.abs(err).max() if err.size else 0.0
    assert l2 <= L2_TOL and mx <= MAX_TOL, f"{what}: L2-rel {l2:.3e}, max-abs {mx:.3e}"
    return l2, mx


def run(sdpa, q, k, v, **kw):
    dev = torch.device("cuda")
    args = [x.to(dev) for x in (q, k, v)]
    if kw.get("mask") is not None:
        kw["mask"] = kw["mask"].to(dev)
    out = sdpa.sdpa_forward(*args, **kw)
    rc, detail = sdpa.sdpa_last_device_status()
    assert rc == 0, f"device status {rc} bits {detail:#x}"
    return out


SMALL = [
    # (B, H, L, D, dtype, causal)
    (1, 4, 128, 64, torch.bfloat16, True),
    (1, 2, 384, 64, torch.bfloat16, True),
    (1, 2, 384, 128, torch.bfloat16, True),
    (2, 1, 200, 128, torch.bfloat16, True),
    (1, 2, 200, 64, torch.float16, False),
    (1, 1, 1, 64, torch.bfloat16, True),
    (1, 1, 2, 128, torch.bfloat16, False),
    (1, 1, 127, 64, torch.float16, True),
    (1, 1, 129, 128, torch.bfloat16, False),
    (1, 2, 1000, 64, torch.bfloat16, True),
    (1, 1, 640, 128, torch.float16, False),
]


@pytest.mark.parametrize("B,H,L,D,dtype,causal", SMALL,
                         ids=[f"{b}x{h}x{l}x{d}-{str(t)[6:]}-{'causal' if c else 'full'}"
                              for b, h, l, d, t, c in SMALL])
def test_small_full(sdpa_lib, B, H, L, D, dtype, causal):
    q, k, v = sdpa_inputs.custom((B, H, L, D), dtype=dtype, seed=100 + L + D)
    out = run(sdpa_lib, q, k, v, is_causal=causal)
    ref = oracle.sdpa(q, k, v, is_causal=causal)
    check(out.double().cpu().numpy(), ref, f"{B}x{H}x{L}x{D}")


@pytest.mark.parametrize("L,D", [(256, 64), (250, 64), (300, 128), (130, 64), (400, 64), (272, 128)])
def test_masked_small(sdpa_lib, L, D):
    q, k, v = sdpa_inputs.custom((1, 2, L, D), dtype=torch.float16, seed=7 + L)
    mask = sdpa_inputs.bernoulli_mask(L, 0.3, seed=50 + L, n_full_rows=5, rows_seed=51 + L)
    full = torch.nonzero(mask.all(dim=1)).flatten()
    assert full.numel() >= 5
    out = run(sdpa_lib, q, k, v, mask=mask)
    ref = oracle.sdpa(q, k, v, mask=mask)
    got = out.double().cpu().numpy()
    check(got, ref, f"masked L={L}")
    assert np.all(got[:, :, full.numpy(), :] == 0.0)


def test_scales(sdpa_lib):
    q, k, v = sdpa_inputs.custom((1, 2, 300, 64), seed=5)
    for s in (0.3, 0.0, -0.2, 1.0):
        out = run(sdpa_lib, q, k, v, is_causal=True, scale=s)
        check(out.double().cpu().numpy(), oracle.sdpa(q, k, v, is_causal=True, scale=s),
              f"scale={s}")


def test_strided_views(sdpa_lib):
    """A [B, L, H, D] buffer consumed as [B, H, L, D] with no copy, and a
    strided output view."""
    B, H, L, D = 2, 3, 257, 64
    base = sdpa_inputs.custom((B, L, H, D), seed=9)
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev).permute(0, 2, 1, 3) for x in base)
    assert not qd.is_contiguous()
    out_buf = torch.full((B, L, H, D), float("nan"), dtype=torch.bfloat16, device=dev)
    out = out_buf.permute(0, 2, 1, 3)
    import scaled_dot_product_forward_gb300 as sdpa
    sdpa.sdpa_forward(qd, kd, vd, out, is_causal=True)
    rc, _ = sdpa.sdpa_last_device_status()
    assert rc == 0
    q, k, v = (x.permute(0, 2, 1, 3) for x in base)
    check(out.double().cpu().numpy(), oracle.sdpa(q, k, v, is_causal=True), "strided")


def test_deterministic(sdpa_lib):
    q, k, v = sdpa_inputs.custom((2, 4, 512, 128), seed=11)
    a = run(sdpa_lib, q, k, v, is_causal=True)
    b = run(sdpa_lib, q, k, v, is_causal=True)
    assert torch.equal(a, b)


def test_rank3_equals_rank4_bitwise(sdpa_lib):
    """Workload 2 as rank-4 [8,16,1024,64] and as rank-3 [128,1024,64]: the
    same fused kernel, identical bits."""
    q, k, v, _ = sdpa_inputs.make(2)
    o4 = run(sdpa_lib, q, k, v, is_causal=True)
    o3 = run(sdpa_lib, q.reshape(128, 1024, 64), k.reshape(128, 1024, 64),
             v.reshape(128, 1024, 64), is_causal=True)
    assert torch.equal(o4.reshape(128, 1024, 64), o3)


def test_one_kernel_per_call(sdpa_lib, tmp_path):
    """The fused path is one GPU kernel per forward (the pages' fused backends
    launch exactly one kernel per forward).  Kernels are counted from the
    profiler's exported trace, which lists every kernel CUPTI saw."""
    import json
    from torch.profiler import ProfilerActivity, profile
    q, k, v = (x.cuda() for x in sdpa_inputs.custom((1, 2, 256, 64), seed=3))
    sdpa_lib.sdpa_forward(q, k, v, is_causal=True)
    torch.cuda.synchronize()
    with profile(activities=[ProfilerActivity.CPU, ProfilerActivity.CUDA]) as prof:
        torch.ones(8, device="cuda").add_(1)  # a torch kernel: shows the profiler sees GPU work
        for _ in range(3):
            sdpa_lib.sdpa_forward(q, k, v, is_causal=True)
        torch.cuda.synchronize()
    path = str(tmp_path / "trace.json")
    prof.export_chrome_trace(path)
    with open(path) as f:
        events = json.load(f)["traceEvents"]
    kernels = [e.get("name", "") for e in events if e.get("cat") == "kernel"]
    if not kernels:
        pytest.skip("the CUDA profiler recorded no kernels at all in this process (not even "
                    "torch's); the ncu launch list is the evidence instead")
    ours = [n for n in kernels if "sdpa_fwd_kernel" in n]
    assert len(ours) == 3, kernels


@pytest.mark.parametrize("kind", ["window", "blockdiag", "none_removed"])
def test_structured_masks(sdpa_lib, kind):
    """Masks with whole tiles free of removed keys (the kernel skips the
    per-element select there) and whole tiles removed."""
    L, D = 640, 64
    q, k, v = sdpa_inputs.custom((1, 2, L, D), dtype=torch.float16, seed=41)
    i = torch.arange(L)
    if kind == "window":          # key j allowed when |i - j| < 100
        mask = (i[:, None] - i[None, :]).abs() >= 100
    elif kind == "blockdiag":     # documents of 200 rows
        mask = (i[:, None] // 200) != (i[None, :] // 200)
    else:
        mask = torch.zeros(L, L, dtype=torch.bool)
    out = run(sdpa_lib, q, k, v, mask=mask)
    check(out.double().cpu().numpy(), oracle.sdpa(q, k, v, mask=mask), kind)


def test_long_sequence_sampled(sdpa_lib):
    """A 131072-long causal sequence: row and tile indices far past 2^16 and
    an L*L far past 2^31, checked on sampled rows (every tile edge would be
    too many for the fp64 oracle)."""
    L, D = 131072, 64
    q, k, v = sdpa_inputs.custom((1, 2, L, D), dtype=torch.bfloat16, seed=81)
    out = run(sdpa_lib, q, k, v, is_causal=True)
    g = torch.Generator().manual_seed(82)
    rows = torch.stack([torch.zeros(40, dtype=torch.long), torch.randint(0, 2, (40,), generator=g),
                        torch.randint(0, L, (40,), generator=g)], 1)
    edge = torch.tensor([[0, h, r] for h in (0, 1) for r in (0, 127, 128, L - 129, L - 128, L - 1)])
    rows = torch.cat([rows, edge])
    ref = oracle.sdpa_rows(q, k, v, rows.numpy(), is_causal=True)
    got = out.cpu()[rows[:, 0], rows[:, 1], rows[:, 2]].double().numpy()
    check(got, ref, "L=131072")

"""Mask tile summary on the GPU (sdpa_mask_tiles) and masked plans, which
launch it before the forward and skip key tiles that remove every key for
both query tiles of a job.  The summary is integer work, so it must match
the oracle's definition bit for bit.  A masked plan's output must equal the
one-shot sdpa_forward's, which reads the mask bytes and visits every tile:
a skipped tile would only have added exact zeros.  Both must match the
fp64 oracle within the parity tolerance."""
import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs
from tests.test_lse import check_lse
from tests.test_parity import check

pytestmark = pytest.mark.gpu


def summary_of(sdpa, mask):
    bits, cls = sdpa.sdpa_mask_tiles(mask.cuda())
    torch.cuda.synchronize()
    return bits.cpu().numpy().view(np.uint32), cls.cpu().numpy()


@pytest.mark.parametrize("L", [1, 100, 128, 300, 400])
def test_summary_matches_oracle(sdpa_lib, L):
    g = torch.Generator().manual_seed(L)
    mask = (torch.rand((L, L), generator=g) < 0.5).to(torch.uint8)
    if L > 128:
        mask[:128, :128] = 0           # a tile that removes nothing
        mask[128:, :128] = 1           # tiles that remove everything
    bits, cls = summary_of(sdpa_lib, mask)
    want_bits, want_cls = oracle.mask_tiles(mask.numpy())
    np.testing.assert_array_equal(bits, want_bits)
    np.testing.assert_array_equal(cls, want_cls)


def test_summary_of_full_size_mask(sdpa_lib):
    """The masked [2048, 2048] Bernoulli(0.3) mask with 16 full rows, on
    sampled tiles against the oracle's definition."""
    w = sdpa_inputs.WORKLOADS[4]
    mask = sdpa_inputs.make(w)[3]
    bits, cls = summary_of(sdpa_lib, mask)
    assert np.all(cls == 1)
    m = mask.numpy()
    for qt, kt in [(0, 0), (3, 11), (15, 15), (7, 2)]:
        sub = m[qt * 128:(qt + 1) * 128, kt * 128:(kt + 1) * 128]
        want_bits, want_cls = oracle.mask_tiles(sub)
        np.testing.assert_array_equal(bits[qt, kt], want_bits[0, 0])


def masks(L):
    i = torch.arange(L)
    return {
        "bernoulli": sdpa_inputs.bernoulli_mask(L, 0.3, seed=51, n_full_rows=3, rows_seed=52),
        "window": ((i[:, None] - i[None, :]).abs() >= 150).to(torch.uint8),
        "blockdiag": ((i[:, None] // 256) != (i[None, :] // 256)).to(torch.uint8),
        # query rows 0..255 remove every key: the first job visits nothing
        "dead_rows": torch.cat([torch.ones(min(256, L), L, dtype=torch.uint8),
                                sdpa_inputs.bernoulli_mask(L, 0.5, seed=53)[min(256, L):]]),
        "causal_as_mask": (i[None, :] > i[:, None]).to(torch.uint8),
    }


CASES = [(1024, 64, torch.float16), (768, 128, torch.bfloat16), (400, 64, torch.bfloat16),
         (272, 128, torch.float16)]


@pytest.mark.parametrize("L,D,dtype", CASES, ids=[f"L{l}-D{d}-{str(t)[6:]}" for l, d, t in CASES])
@pytest.mark.parametrize("kind", ["bernoulli", "window", "blockdiag", "dead_rows",
                                  "causal_as_mask"])
def test_masked_plan(sdpa_lib, L, D, dtype, kind):
    mask = masks(L)[kind]
    q, k, v = sdpa_inputs.custom((2, 2, L, D), dtype=dtype, seed=L + D)
    qd, kd, vd, md = (x.cuda() for x in (q, k, v, mask))
    one_shot = sdpa_lib.sdpa_forward(qd, kd, vd, mask=md)
    out = torch.full_like(qd, float("nan"))
    lse = torch.full(q.shape[:-1], float("nan"), dtype=torch.float32, device="cuda")
    plan = sdpa_lib.SdpaPlan(qd, kd, vd, out, mask=md)
    plan.set_lse(lse)
    for _ in range(2):               # the summary is rebuilt on every launch
        plan.launch()
    torch.cuda.synchronize()
    rc, detail = sdpa_lib.sdpa_last_device_status()
    assert rc == 0, f"device status {rc} bits {detail:#x}"
    plan.close()
    assert torch.equal(out, one_shot), f"{kind}: plan differs from the one-shot call"
    ref, ref_lse = oracle.sdpa(q, k, v, mask=mask, return_lse=True)
    check(out.double().cpu().numpy(), ref, kind)
    check_lse(lse.cpu().numpy(), ref_lse)
    if kind == "dead_rows":
        assert torch.all(out[:, :, :256] == 0)


def test_plan_follows_mask_contents(sdpa_lib):
    """The summary is rebuilt from the mask on each launch: change the mask
    in place between launches and the output follows."""
    L, D = 512, 64
    q, k, v = sdpa_inputs.custom((1, 2, L, D), dtype=torch.float16, seed=61)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    md = masks(L)["window"].cuda()
    out = torch.empty_like(qd)
    plan = sdpa_lib.SdpaPlan(qd, kd, vd, out, mask=md)
    plan.launch()
    first = out.clone()
    md.copy_(masks(L)["blockdiag"].cuda())
    plan.launch()
    torch.cuda.synchronize()
    plan.close()
    assert torch.equal(first, sdpa_lib.sdpa_forward(qd, kd, vd, mask=masks(L)["window"].cuda()))
    check(out.double().cpu().numpy(), oracle.sdpa(q, k, v, mask=masks(L)["blockdiag"]),
          "after the mask changed")


def test_masked_workload_plan_sampled(sdpa_lib):
    """The masked [2, 16, 2048, 64] fp16 workload through a plan (the
    launch the benchmark's plan mode times): equal to the one-shot call."""
    w = sdpa_inputs.WORKLOADS[4]
    q, k, v, mask = sdpa_inputs.make(w)
    qd, kd, vd, md = (x.cuda() for x in (q, k, v, mask))
    out = torch.empty_like(qd)
    plan = sdpa_lib.SdpaPlan(qd, kd, vd, out, mask=md)
    plan.launch()
    torch.cuda.synchronize()
    plan.close()
    assert torch.equal(out, sdpa_lib.sdpa_forward(qd, kd, vd, mask=md))
    assert torch.all(out[:, :, sdpa_inputs.full_rows(w)] == 0)


def test_masked_plan_rank3_unaligned_length(sdpa_lib):
    """Rank-3 [H, L, D] with L = 300: the mask rows are not 16-byte multiples,
    so the summary kernel reads bytes one at a time, and the last tiles are
    ragged in both rows and keys."""
    L, D = 300, 64
    i = torch.arange(L)
    mask = ((i[:, None] - i[None, :]).abs() >= 90).to(torch.uint8)
    mask[:40] = 1                                   # rows with every key removed
    q, k, v = sdpa_inputs.custom((3, L, D), dtype=torch.bfloat16, seed=77)
    qd, kd, vd, md = (x.cuda() for x in (q, k, v, mask))
    out = torch.full_like(qd, float("nan"))
    plan = sdpa_lib.SdpaPlan(qd, kd, vd, out, mask=md)
    plan.launch()
    torch.cuda.synchronize()
    plan.close()
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    assert torch.equal(out, sdpa_lib.sdpa_forward(qd, kd, vd, mask=md))
    assert torch.all(out[:, :40] == 0)
    check(out.double().cpu().numpy(), oracle.sdpa(q, k, v, mask=mask), "rank-3 L=300")


def test_masked_plan_rebinds_to_another_mask(sdpa_lib):
    """set_pointers moves a masked plan to another mask buffer: its summary
    is rebuilt from the new mask on the next launch."""
    L, D = 512, 128
    q, k, v = sdpa_inputs.custom((1, 2, L, D), dtype=torch.bfloat16, seed=78)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    m1, m2 = masks(L)["blockdiag"].cuda(), masks(L)["dead_rows"].cuda()
    out = torch.empty_like(qd)
    plan = sdpa_lib.SdpaPlan(qd, kd, vd, out, mask=m1)
    plan.launch()
    first = out.clone()
    plan.set_pointers(qd, kd, vd, out, mask=m2)
    plan.launch()
    torch.cuda.synchronize()
    plan.close()
    assert torch.equal(first, sdpa_lib.sdpa_forward(qd, kd, vd, mask=m1))
    assert torch.equal(out, sdpa_lib.sdpa_forward(qd, kd, vd, mask=m2))


def test_masked_plan_visits_across_chunks(sdpa_lib):
    """L = 4224: 33 key tiles, so the visited-tile cursor spans two 32-tile
    chunks, with skipped tiles on both sides of the chunk edge and a job in
    the second chunk that visits nothing."""
    L, D = 4224, 64
    i = torch.arange(L)
    mask = ((i[:, None] - i[None, :]).abs() >= 300).to(torch.uint8)
    mask[4096:] = 1                                  # the last query tile removes every key
    q, k, v = sdpa_inputs.custom((1, 2, L, D), dtype=torch.float16, seed=79)
    qd, kd, vd, md = (x.cuda() for x in (q, k, v, mask))
    bits, cls = summary_of(sdpa_lib, mask)
    assert cls.shape == (33, 33) and (cls == 2).sum() > 0 and cls[32].tolist() == [2] * 33
    out = torch.empty_like(qd)
    plan = sdpa_lib.SdpaPlan(qd, kd, vd, out, mask=md)
    plan.launch()
    torch.cuda.synchronize()
    plan.close()
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    assert torch.equal(out, sdpa_lib.sdpa_forward(qd, kd, vd, mask=md))
    assert torch.all(out[:, :, 4096:] == 0)
    g = torch.Generator().manual_seed(80)
    rows = torch.stack([torch.zeros(96, dtype=torch.long), torch.randint(0, 2, (96,), generator=g),
                        torch.randint(0, L, (96,), generator=g)], 1)
    edge = torch.tensor([[0, 1, r] for r in (0, 4095, 4096, 4223, 3967, 3968)])
    rows = torch.cat([rows, edge])
    ref = oracle.sdpa_rows(q, k, v, rows.numpy(), mask=mask)
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]].double().cpu().numpy()
    check(got, ref, "33 tiles")

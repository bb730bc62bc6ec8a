"""Sparse top-k attention and its index preparation on the GPU, against the
fp64 oracle (``oracle.sdpa_sparse``, ``oracle.sparse_compact_indices``).
Index work is compared bit for bit; outputs at L2-relative <= 1e-2 and
max-abs <= 2e-2, lse to 2e-3."""
import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs

pytestmark = pytest.mark.gpu

L2_TOL, MAX_TOL = 1e-2, 2e-2


def check(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = got - ref
    l2 = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    assert l2 <= L2_TOL and mx <= MAX_TOL, f"{what}: L2-rel {l2:.3e}, max-abs {mx:.3e}"


def make(total_q, total_k, H, D, topk, dtype, seed, empty_rows=True):
    q = sdpa_inputs.custom((total_q, H, D), dtype=dtype, seed=seed)[0]
    k, v = (x[:, 0].contiguous() for x in sdpa_inputs.custom((total_k, 1, D), dtype=dtype,
                                                                seed=seed + 1)[:2])
    rng = np.random.default_rng(seed)
    idx = np.stack([rng.choice(total_k, topk, replace=False) for _ in range(total_q)]).astype(np.int32)
    length = rng.integers(0, topk + 1, size=total_q).astype(np.int32)
    length[0] = topk
    if total_q > 2:
        length[1] = 1
        length[2] = 0 if empty_rows else 5
    return q, k, v, idx, length


CASES = [  # total_q, total_k, H, D, topk, dtype
    (40, 3000, 128, 128, 300, torch.bfloat16),
    (15, 700, 160, 128, 300, torch.bfloat16),   # two head groups: 128 and 32
    (33, 2000, 64, 128, 1000, torch.bfloat16),
    (50, 1500, 16, 64, 257, torch.float16),
    (20, 900, 192, 64, 128, torch.bfloat16),
]


@pytest.mark.parametrize("case", CASES, ids=[f"q{c[0]}-k{c[1]}-H{c[2]}-D{c[3]}-topk{c[4]}" for c in CASES])
def test_sparse_matches_oracle(sdpa_lib, case):
    total_q, total_k, H, D, topk, dtype = case
    q, k, v, idx, length = make(*case, seed=1200 + H + D)
    dev = torch.device("cuda")
    out, lse = sdpa_lib.sdpa_sparse_forward(
        q.to(dev), k.to(dev), v.to(dev), torch.from_numpy(idx).to(dev),
        torch.from_numpy(length).to(dev), return_lse=True)
    rc, detail = sdpa_lib.sdpa_last_device_status()
    assert rc == 0, f"device status bits {detail:#x}"
    ref, ref_lse = oracle.sdpa_sparse(q, k, v, idx, topk_length=length, return_lse=True)
    check(out.double().cpu().numpy(), ref, "out")
    got_lse = lse.double().cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got_lse), fin)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=0, atol=2e-3)
    assert np.all(out.cpu()[2].float().numpy() == 0.0)   # the row with no key


def test_out_of_range_entries_are_removed(sdpa_lib):
    q, k, v, idx, length = make(16, 500, 128, 128, 200, torch.bfloat16, seed=1300)
    idx[:, 7] = -5
    idx[:, 11] = 500 + 3
    dev = torch.device("cuda")
    out = sdpa_lib.sdpa_sparse_forward(q.to(dev), k.to(dev), v.to(dev),
                                       torch.from_numpy(idx).to(dev),
                                       torch.from_numpy(length).to(dev))
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    # reference: the same rows without those entries
    keep = [[x for t, x in enumerate(r[:n]) if 0 <= x < 500] for r, n in zip(idx, length)]
    n2 = np.array([len(r) for r in keep])
    idx2 = np.zeros_like(idx)
    for i, r in enumerate(keep):
        idx2[i, :len(r)] = r
    check(out.double().cpu().numpy(), oracle.sdpa_sparse(q, k, v, idx2, topk_length=n2), "removed")


def test_all_keys_equals_dense_full_attention(sdpa_lib):
    """Every key in order: the sparse path computes the same tiles in the same
    order as the dense kernel does for one head against the shared K/V."""
    L, H, D = 512, 128, 128
    q = sdpa_inputs.custom((L, H, D), seed=1310)[0]
    k, v = (x[:, 0].contiguous() for x in sdpa_inputs.custom((L, 1, D), seed=1311)[:2])
    dev = torch.device("cuda")
    idx = torch.arange(L, dtype=torch.int32).repeat(L, 1)
    out = sdpa_lib.sdpa_sparse_forward(q.to(dev), k.to(dev), v.to(dev), idx.to(dev))
    kk, vv = (x.to(dev)[None].expand(H, L, D).contiguous() for x in (k, v))
    dense = sdpa_lib.sdpa_forward(q.to(dev).permute(1, 0, 2), kk, vv)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    diff = (out.permute(1, 0, 2).float() - dense.float()).abs().max().item()
    assert diff <= 2e-2, diff
    check(out.double().cpu().numpy(),
          oracle.sdpa_sparse(q, k, v, idx.numpy()), "all keys")


@pytest.mark.parametrize("causal", [True, False])
def test_compaction_bit_exact(sdpa_lib, causal):
    rng = np.random.default_rng(77)
    cu_q = np.array([0, 40, 40, 130, 300], dtype=np.int32)
    cu_k = np.array([0, 50, 64, 200, 333], dtype=np.int32)
    total_q, topk = 300, 96
    idx_local = rng.integers(-2, 180, size=(total_q, topk)).astype(np.int32)
    dev = torch.device("cuda")
    g, n = sdpa_lib.sdpa_sparse_compact(torch.from_numpy(idx_local).to(dev),
                                        torch.from_numpy(cu_q).to(dev),
                                        torch.from_numpy(cu_k).to(dev), is_causal=causal)
    ref_g, ref_n = oracle.sparse_compact_indices(idx_local, cu_q, cu_k, is_causal=causal)
    np.testing.assert_array_equal(n.cpu().numpy(), ref_n)
    np.testing.assert_array_equal(g.cpu().numpy(), ref_g)


def test_compaction_then_forward(sdpa_lib):
    rng = np.random.default_rng(78)
    cu = np.array([0, 130, 260, 700], dtype=np.int32)
    total, H, D, topk = 700, 64, 128, 200
    q = sdpa_inputs.custom((total, H, D), seed=1320)[0]
    k, v = (x[:, 0].contiguous() for x in sdpa_inputs.custom((total, 1, D), seed=1321)[:2])
    idx_local = rng.integers(-1, 440, size=(total, topk)).astype(np.int32)
    dev = torch.device("cuda")
    cud = torch.from_numpy(cu).to(dev)
    g, n = sdpa_lib.sdpa_sparse_compact(torch.from_numpy(idx_local).to(dev), cud, cud)
    out = sdpa_lib.sdpa_sparse_forward(q.to(dev), k.to(dev), v.to(dev), g, n)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    ref_g, ref_n = oracle.sparse_compact_indices(idx_local, cu, cu, is_causal=True)
    check(out.double().cpu().numpy(), oracle.sdpa_sparse(q, k, v, ref_g, topk_length=ref_n),
          "compact + forward")


def test_one_kv_tensor_for_keys_and_values(sdpa_lib):
    """The same tensor as k and v (one kv tensor, gathered once)."""
    q, kv, _, idx, length = make(48, 1024, 64, 128, 384, torch.bfloat16, seed=1330)
    dev = torch.device("cuda")
    kvd = kv.to(dev)
    out, lse = sdpa_lib.sdpa_sparse_forward(q.to(dev), kvd, kvd, torch.from_numpy(idx).to(dev),
                                            torch.from_numpy(length).to(dev), return_lse=True)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    ref, ref_lse = oracle.sdpa_sparse(q, kv, kv, idx, topk_length=length, return_lse=True)
    check(out.double().cpu().numpy(), ref, "one kv tensor")
    # and identical to passing a copy as v
    out2 = sdpa_lib.sdpa_sparse_forward(q.to(dev), kvd, kvd.clone(),
                                        torch.from_numpy(idx).to(dev),
                                        torch.from_numpy(length).to(dev))
    assert torch.equal(out, out2)


HALF_ROW_CASES = [  # total_q, total_k, H, D, topk, dtype -- groups of at most 64 heads
    (1, 500, 64, 128, 300, torch.bfloat16),    # one row
    (7, 800, 48, 128, 200, torch.float16),     # the last quarter of the tile holds no head
    (9, 700, 20, 128, 150, torch.bfloat16),    # a quarter holds 4 of its 16 heads
    (5, 300, 8, 64, 100, torch.float16),       # fewer heads than one quarter
    (29, 1200, 32, 64, 640, torch.bfloat16),   # head size 64, ragged last tiles
    (6, 5000, 64, 128, 4100, torch.bfloat16),  # 33 key tiles a row: many laps of the ring
]


@pytest.mark.parametrize("case", HALF_ROW_CASES,
                         ids=[f"q{c[0]}-k{c[1]}-H{c[2]}-D{c[3]}-topk{c[4]}" for c in HALF_ROW_CASES])
def test_half_row_form_matches_oracle(sdpa_lib, case):
    """Groups of at most 64 heads run M = 64 products (16 heads in each
    quarter of TMEM) and split every row's keys between two softmax threads."""
    total_q, total_k, H, D, topk, dtype = case
    q, k, v, idx, length = make(*case, seed=1400 + H + D + total_q)
    dev = torch.device("cuda")
    out, lse = sdpa_lib.sdpa_sparse_forward(
        q.to(dev), k.to(dev), v.to(dev), torch.from_numpy(idx).to(dev),
        torch.from_numpy(length).to(dev), return_lse=True)
    rc, detail = sdpa_lib.sdpa_last_device_status()
    assert rc == 0, f"device status bits {detail:#x}"
    ref, ref_lse = oracle.sdpa_sparse(q, k, v, idx, topk_length=length, return_lse=True)
    check(out.double().cpu().numpy(), ref, "out")
    got_lse = lse.double().cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got_lse), fin)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=0, atol=2e-3)
    if total_q > 2:
        assert np.all(out.cpu()[2].float().numpy() == 0.0)   # the row with no key


def test_rows_do_not_depend_on_their_schedule(sdpa_lib):
    """Dropping the first query row hands every other row to another CTA and
    position in its job list: each row's output must stay bit-identical."""
    q, kv, _, idx, length = make(41, 1500, 64, 128, 700, torch.bfloat16, seed=1410)
    dev = torch.device("cuda")
    qd, kvd = q.to(dev), kv.to(dev)
    idd, lnd = torch.from_numpy(idx).to(dev), torch.from_numpy(length).to(dev)
    full = sdpa_lib.sdpa_sparse_forward(qd, kvd, kvd, idd, lnd)
    tail = sdpa_lib.sdpa_sparse_forward(qd[1:].contiguous(), kvd, kvd, idd[1:].contiguous(),
                                        lnd[1:].contiguous())
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    assert torch.equal(full[1:], tail)


def test_negative_scale(sdpa_lib):
    """A negative scale makes the row minimum the stabiliser."""
    q, k, v, idx, length = make(12, 600, 64, 128, 256, torch.bfloat16, seed=1420)
    dev = torch.device("cuda")
    out = sdpa_lib.sdpa_sparse_forward(q.to(dev), k.to(dev), v.to(dev),
                                       torch.from_numpy(idx).to(dev),
                                       torch.from_numpy(length).to(dev), scale=-0.2)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    check(out.double().cpu().numpy(),
          oracle.sdpa_sparse(q, k, v, idx, topk_length=length, scale=-0.2), "negative scale")


ONE_KV_CASES = [  # total_q, total_k, H, D, topk, dtype -- one tensor as keys and values
    (21, 1400, 128, 128, 520, torch.bfloat16),  # more than 64 heads: M = 128 products
    (17, 900, 48, 64, 300, torch.float16),      # head size 64, half-row form
]


@pytest.mark.parametrize("case", ONE_KV_CASES,
                         ids=[f"q{c[0]}-k{c[1]}-H{c[2]}-D{c[3]}-topk{c[4]}" for c in ONE_KV_CASES])
def test_one_kv_tensor_matches_oracle(sdpa_lib, case):
    """One kv tensor (rows gathered once into a deeper ring) on the paths
    the benchmark workload does not take."""
    total_q, total_k, H, D, topk, dtype = case
    q, kv, _, idx, length = make(*case, seed=1440 + H + D)
    dev = torch.device("cuda")
    kvd = kv.to(dev)
    out, lse = sdpa_lib.sdpa_sparse_forward(q.to(dev), kvd, kvd, torch.from_numpy(idx).to(dev),
                                            torch.from_numpy(length).to(dev), return_lse=True)
    assert sdpa_lib.sdpa_last_device_status()[0] == 0
    ref, ref_lse = oracle.sdpa_sparse(q, kv, kv, idx, topk_length=length, return_lse=True)
    check(out.double().cpu().numpy(), ref, "one kv tensor")
    got_lse = lse.double().cpu().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got_lse), fin)
    np.testing.assert_allclose(got_lse[fin], ref_lse[fin], rtol=0, atol=2e-3)

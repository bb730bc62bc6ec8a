"""Pins for the sparse top-k oracle (``oracle.sdpa_sparse``) and its index
preparation (``oracle.sparse_compact_indices``), against formulations that
share none of their code: the dense C oracle (all keys in order equals
full attention; keys 0..i equals causal attention), closed forms and
invariants."""
import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs


def test_all_keys_in_order_equals_dense():
    L, H, D = 33, 3, 8
    q = sdpa_inputs.custom((L, H, D), dtype=torch.float64, seed=81)[0]
    k, v = (x[:, 0] for x in sdpa_inputs.custom((L, 1, D), dtype=torch.float64, seed=82)[:2])
    idx = np.tile(np.arange(L), (L, 1))
    got, lse = oracle.sdpa_sparse(q, k, v, idx, return_lse=True)
    # dense: every head against the one shared key/value head
    kk, vv = (x[None].expand(H, L, D).contiguous() for x in (k, v))
    ref, ref_lse = oracle.sdpa(q.permute(1, 0, 2), kk, vv, return_lse=True)
    np.testing.assert_allclose(got, ref.transpose(1, 0, 2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse.T, rtol=0, atol=1e-12)


def test_prefix_keys_equals_causal():
    L, H, D = 20, 2, 4
    q = sdpa_inputs.custom((L, H, D), dtype=torch.float64, seed=83)[0]
    k, v = (x[:, 0] for x in sdpa_inputs.custom((L, 1, D), dtype=torch.float64, seed=84)[:2])
    idx = np.tile(np.arange(L), (L, 1))       # row i uses keys 0..i via its length
    got = oracle.sdpa_sparse(q, k, v, idx, topk_length=np.arange(1, L + 1))
    kk, vv = (x[None].expand(H, L, D).contiguous() for x in (k, v))
    ref = oracle.sdpa(q.permute(1, 0, 2), kk, vv, is_causal=True)
    np.testing.assert_allclose(got, ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_one_key_and_empty_rows():
    q = sdpa_inputs.custom((4, 2, 8), dtype=torch.float64, seed=85)[0]
    k, v = (x[:, 0] for x in sdpa_inputs.custom((9, 1, 8), dtype=torch.float64, seed=86)[:2])
    idx = np.array([[7, 1], [3, 3], [0, 5], [2, 2]])
    out, lse = oracle.sdpa_sparse(q, k, v, idx, topk_length=[1, 1, 0, 1], return_lse=True)
    np.testing.assert_array_equal(out[0], np.tile(v.numpy()[7], (2, 1)))
    np.testing.assert_array_equal(out[2], 0.0)
    assert np.all(np.isneginf(lse[2]))
    # one key: lse = scale * q . k
    np.testing.assert_allclose(lse[3], (q[3].numpy() @ k.numpy()[2]) / np.sqrt(8), atol=1e-14)


def test_entry_order_does_not_matter():
    q = sdpa_inputs.custom((5, 2, 8), dtype=torch.float64, seed=87)[0]
    k, v = (x[:, 0] for x in sdpa_inputs.custom((30, 1, 8), dtype=torch.float64, seed=88)[:2])
    rng = np.random.default_rng(3)
    idx = np.stack([rng.choice(30, 12, replace=False) for _ in range(5)])
    a = oracle.sdpa_sparse(q, k, v, idx)
    b = oracle.sdpa_sparse(q, k, v, idx[:, ::-1].copy())
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


def test_compaction_closed_forms():
    # one document of 6 queries and 6 keys; row i lists keys 0..5
    idx = np.tile(np.arange(6), (6, 1))
    g, n = oracle.sparse_compact_indices(idx, [0, 6], [0, 6], is_causal=True)
    np.testing.assert_array_equal(n, np.arange(1, 7))          # keys 0..i survive
    for i in range(6):
        np.testing.assert_array_equal(g[i, :i + 1], np.arange(i + 1))
        assert np.all(g[i, i + 1:] == -1)
    g, n = oracle.sparse_compact_indices(np.full((6, 4), -1), [0, 6], [0, 6])
    assert np.all(n == 0) and np.all(g == -1)


def test_compaction_matches_vectorised_form():
    """Against a numpy formulation (boolean validity, stable order by column)."""
    rng = np.random.default_rng(9)
    cu_q = np.array([0, 7, 7, 20, 31])
    cu_k = np.array([0, 9, 12, 25, 40])
    total_q, topk = 31, 10
    idx = rng.integers(-3, 14, size=(total_q, topk))
    for causal in (False, True):
        g, n = oracle.sparse_compact_indices(idx, cu_q, cu_k, is_causal=causal)
        doc = np.searchsorted(cu_q, np.arange(total_q), side="right") - 1
        pos = np.arange(total_q) - cu_q[doc]
        nk = (cu_k[1:] - cu_k[:-1])[doc]
        valid = (idx >= 0) & (idx < nk[:, None])
        if causal:
            valid &= idx <= pos[:, None]
        np.testing.assert_array_equal(n, valid.sum(1))
        for i in range(total_q):
            want = idx[i][valid[i]] + cu_k[doc[i]]
            np.testing.assert_array_equal(g[i, :n[i]], want)
            assert np.all(g[i, n[i]:] == -1)

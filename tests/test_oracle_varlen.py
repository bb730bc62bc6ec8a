"""Pins for the packed-document oracle (``oracle.sdpa_varlen``), checked
against formulations that share none of its slicing: the dense oracle over
the whole packed axis with a block-diagonal mask, and closed forms."""
import math

import numpy as np
import pytest
import torch

import oracle
import sdpa_inputs


def block_mask(cu, total, causal):
    """[total, total] bytes, 1 = removed: keys outside the query's document
    (and, causally, keys after the query)."""
    doc = np.full(total, -1)
    for i, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        doc[a:b] = i
    m = doc[:, None] != doc[None, :]
    if causal:
        m |= np.arange(total)[None, :] > np.arange(total)[:, None]
    return torch.from_numpy(m.astype(np.uint8))


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_block_diagonal_mask(causal):
    cu = [0, 5, 5, 17, 18, 40]          # includes an empty and a one-token document
    total, H, D = 40, 2, 8
    q, k, v = sdpa_inputs.custom((total, H, D), dtype=torch.float64, seed=71)
    got = oracle.sdpa_varlen(q, k, v, cu, is_causal=causal)
    m = block_mask(np.array(cu), total, causal)
    # dense over the packed axis: [total, H, D] -> [H, total, D]
    ref = oracle.sdpa(q.permute(1, 0, 2), k.permute(1, 0, 2), v.permute(1, 0, 2), mask=m)
    np.testing.assert_allclose(got, ref.transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_single_token_documents_return_their_value_row():
    total, H, D = 6, 3, 4
    q, k, v = sdpa_inputs.custom((total, H, D), dtype=torch.float64, seed=72)
    cu = list(range(total + 1))
    out, lse = oracle.sdpa_varlen(q, k, v, cu, is_causal=False, return_lse=True)
    np.testing.assert_array_equal(out, v.numpy())
    # one admissible key: lse = scale * q . k
    s = (q * k).sum(-1).numpy() / math.sqrt(D)
    np.testing.assert_allclose(lse, s.T, rtol=0, atol=1e-14)


def test_rows_outside_every_document_are_nan():
    q, k, v = sdpa_inputs.custom((10, 1, 4), dtype=torch.float64, seed=73)
    out = oracle.sdpa_varlen(q, k, v, [2, 5, 7], is_causal=True)
    assert np.isnan(out[:2]).all() and np.isnan(out[7:]).all()
    assert np.isfinite(out[2:7]).all()


@pytest.mark.parametrize("cu", [[0, 4, 3], [-1, 4], [0, 11]])
def test_bad_offsets_rejected(cu):
    q, k, v = sdpa_inputs.custom((10, 1, 4), dtype=torch.float64, seed=74)
    with pytest.raises(ValueError):
        oracle.sdpa_varlen(q, k, v, cu)

"""Pins for the fp64 oracle: checks against facts that do not come from the
oracle itself.  Each pin takes ``impl(q, k, v, mask=None, is_causal=False,
scale=None) -> ndarray`` so the same checks also run against deliberately
broken builds of the oracle source (``test_oracle_mutants.py``).

Sources of truth used here:
  * brute force in 40-digit decimal arithmetic, written independently: the
    softmax is evaluated as exp(s_j) / sum exp(s) directly (no max shift),
    over the admissible keys only;
  * closed forms of the definition (five steps of the NaiveCausalAttention
    module in "Profiling attention in PyTorch: kernels, backends and where the
    time goes", news.bpdata.com, section "Naiv causal attention"):
    causal row 0 -> v[0]; q = 0 or scale = 0 -> mean of the admissible v rows;
    a single admissible key j -> v[j]; all keys equal -> mean of admissible v;
    a fully removed row -> zeros (safe softmax of the math backend, same page,
    "Math backend" section);
  * invariants: attention weights sum to one (v = 1 -> out = 1), linearity in
    v, joint permutation of keys and values (non-causal), shifting every key by
    one vector c (each row's scores move by the constant q.c);
  * torch's CPU math backend in fp64, the backend that page calls the correct,
    NaN-safe reference (its boolean attn_mask means True = attend, so the mask
    is inverted for it);
  * for the log-sum-exp output (the log of the softmax denominator): decimal
    brute force, closed forms (q = 0 -> log of the number of admissible keys,
    one admissible key -> its scaled score, no admissible key -> -inf) and
    torch.logsumexp over explicitly computed, masked scores.
"""
from __future__ import annotations

from decimal import Decimal, getcontext

import numpy as np


def _rng(seed):
    return np.random.default_rng(seed)


def brute_force_decimal(q, k, v, mask=None, is_causal=False, scale=None):
    """Per-element attention in 40-digit decimals.  q, k, v: [H, L, D]."""
    getcontext().prec = 40
    H, L, D = q.shape
    sc = Decimal(float(1.0 / np.sqrt(D) if scale is None else scale))
    out = np.zeros((H, L, D))
    for h in range(H):
        for i in range(L):
            keys = [j for j in range(L)
                    if not (is_causal and j > i) and not (mask is not None and mask[i, j])]
            if not keys:
                continue  # safe softmax: zero row
            w = {}
            for j in keys:
                dot = sum(Decimal(float(q[h, i, d])) * Decimal(float(k[h, j, d])) for d in range(D))
                w[j] = (dot * sc).exp()
            z = sum(w.values())
            for d in range(D):
                out[h, i, d] = float(sum(w[j] * Decimal(float(v[h, j, d])) for j in keys) / z)
    return out


def _tiny_cases():
    g = _rng(7)
    cases = []
    for (H, L, D) in [(1, 1, 1), (2, 3, 2), (1, 9, 4), (2, 7, 3), (1, 5, 4)]:
        q, k, v = (g.standard_normal((H, L, D)) for _ in range(3))
        mask = g.random((L, L)) < 0.4
        if L > 2:
            mask[1, :] = True  # one fully removed row
        cases.append((q, k, v, None, False, None))
        cases.append((q, k, v, None, True, None))
        cases.append((q, k, v, mask, False, None))
        cases.append((q, k, v, None, True, 0.37))
    return cases


def pin_brute_force(impl):
    for (q, k, v, mask, causal, scale) in _tiny_cases():
        got = impl(q, k, v, mask=mask, is_causal=causal, scale=scale)
        ref = brute_force_decimal(q, k, v, mask, causal, scale)
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def pin_causal_row0(impl):
    g = _rng(11)
    q, k, v = (g.standard_normal((2, 6, 8)) for _ in range(3))
    out = impl(q, k, v, is_causal=True)
    # softmax over a single admissible score is exactly 1
    assert np.array_equal(out[:, 0, :], v[:, 0, :])


def pin_zero_query_prefix_mean(impl):
    g = _rng(12)
    H, L, D = 2, 7, 5
    q = np.zeros((H, L, D))
    k, v = g.standard_normal((H, L, D)), g.standard_normal((H, L, D))
    out = impl(q, k, v, is_causal=True)
    pref = np.cumsum(v, axis=1) / np.arange(1, L + 1)[None, :, None]
    np.testing.assert_allclose(out, pref, rtol=0, atol=1e-14)
    out_nc = impl(q, k, v, is_causal=False)
    np.testing.assert_allclose(out_nc, np.broadcast_to(v.mean(axis=1, keepdims=True), v.shape),
                               rtol=0, atol=1e-14)


def pin_zero_scale_mean(impl):
    g = _rng(13)
    q, k, v = (g.standard_normal((1, 6, 3)) for _ in range(3))
    mask = g.random((6, 6)) < 0.5
    np.fill_diagonal(mask, False)
    out = impl(q, k, v, mask=mask, scale=0.0)
    for i in range(6):
        keep = ~mask[i]
        np.testing.assert_allclose(out[0, i], v[0, keep].mean(axis=0), rtol=0, atol=1e-14)


def pin_single_key(impl):
    g = _rng(14)
    L = 6
    q, k, v = (g.standard_normal((2, L, 4)) for _ in range(3))
    perm = g.permutation(L)
    mask = np.ones((L, L), dtype=bool)
    mask[np.arange(L), perm] = False  # row i may only see key perm[i]
    out = impl(q, k, v, mask=mask)
    assert np.array_equal(out, v[:, perm, :])


def pin_equal_keys(impl):
    g = _rng(15)
    H, L, D = 1, 8, 4
    q = g.standard_normal((H, L, D))
    k = np.repeat(g.standard_normal((H, 1, D)), L, axis=1)
    v = g.standard_normal((H, L, D))
    out = impl(q, k, v, is_causal=True)
    pref = np.cumsum(v, axis=1) / np.arange(1, L + 1)[None, :, None]
    np.testing.assert_allclose(out, pref, rtol=0, atol=1e-14)


def pin_fully_masked_rows_zero(impl):
    g = _rng(16)
    L = 7
    q, k, v = (g.standard_normal((1, L, 4)) for _ in range(3))
    mask = g.random((L, L)) < 0.3
    mask[[0, 3, 6], :] = True
    out = impl(q, k, v, mask=mask)
    assert np.all(np.isfinite(out))
    assert np.array_equal(out[0, [0, 3, 6]], np.zeros((3, 4)))
    assert np.all(np.abs(out[0, [1, 2, 4, 5]]).sum(axis=1) > 0)


def pin_weights_sum_to_one(impl):
    g = _rng(17)
    L = 9
    q, k = g.standard_normal((2, L, 4)) * 3, g.standard_normal((2, L, 4)) * 3
    ones = np.ones((2, L, 4))
    for causal, mask in [(True, None), (False, None), (False, g.random((L, L)) < 0.5)]:
        if mask is not None:
            mask[:, 0] = False
        out = impl(q, k, ones, mask=mask, is_causal=causal)
        np.testing.assert_allclose(out, ones, rtol=0, atol=1e-14)


def pin_linearity_in_v(impl):
    g = _rng(18)
    q, k, v1, v2 = (g.standard_normal((2, 8, 4)) for _ in range(4))
    a, b = 1.75, -0.5
    lhs = impl(q, k, a * v1 + b * v2, is_causal=True)
    rhs = a * impl(q, k, v1, is_causal=True) + b * impl(q, k, v2, is_causal=True)
    np.testing.assert_allclose(lhs, rhs, rtol=0, atol=1e-13)


def pin_permutation_invariance(impl):
    g = _rng(19)
    L = 8
    q, k, v = (g.standard_normal((2, L, 4)) for _ in range(3))
    mask = g.random((L, L)) < 0.3
    perm = g.permutation(L)
    base = impl(q, k, v, mask=mask)
    moved = impl(q, k[:, perm], v[:, perm], mask=mask[:, perm])
    np.testing.assert_allclose(base, moved, rtol=0, atol=1e-13)


def pin_key_shift_invariance(impl):
    g = _rng(20)
    q, k, v = (g.standard_normal((2, 8, 4)) for _ in range(3))
    c = g.standard_normal((1, 1, 4))
    base = impl(q, k, v, is_causal=True)
    shifted = impl(q, k + c, v, is_causal=True)
    np.testing.assert_allclose(base, shifted, rtol=0, atol=1e-12)


def pin_torch_math_backend(impl):
    import torch
    import torch.nn.functional as F
    from torch.nn.attention import SDPBackend, sdpa_kernel

    g = _rng(21)
    for (B, H, L, D) in [(1, 2, 5, 4), (2, 3, 17, 8), (1, 2, 64, 16)]:
        q, k, v = (g.standard_normal((B, H, L, D)) for _ in range(3))
        mask = g.random((L, L)) < 0.3
        mask[:, 0] = False  # keep every row admissible: compare full rows only
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        with sdpa_kernel(SDPBackend.MATH):
            ref_c = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True).numpy()
            ref_m = F.scaled_dot_product_attention(
                tq, tk, tv, attn_mask=torch.from_numpy(~mask)).numpy()
            ref_s = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=0.3).numpy()
        np.testing.assert_allclose(impl(q, k, v, is_causal=True), ref_c, rtol=0, atol=1e-12)
        np.testing.assert_allclose(impl(q, k, v, mask=mask), ref_m, rtol=0, atol=1e-12)
        np.testing.assert_allclose(impl(q, k, v, is_causal=True, scale=0.3), ref_s,
                                   rtol=0, atol=1e-12)


def _lse_impl(impl):
    """The pins call impl(q, k, v, ...); LSE pins need its second output."""
    def f(q, k, v, **kw):
        return impl(q, k, v, return_lse=True, **kw)[1]
    return f


def brute_force_lse_decimal(q, k, mask=None, is_causal=False, scale=None):
    getcontext().prec = 40
    H, L, D = q.shape
    sc = Decimal(float(1.0 / np.sqrt(D) if scale is None else scale))
    out = np.zeros((H, L))
    for h in range(H):
        for i in range(L):
            keys = [j for j in range(L)
                    if not (is_causal and j > i) and not (mask is not None and mask[i, j])]
            if not keys:
                out[h, i] = -np.inf
                continue
            z = sum((sum(Decimal(float(q[h, i, d])) * Decimal(float(k[h, j, d]))
                         for d in range(D)) * sc).exp() for j in keys)
            out[h, i] = float(z.ln())
    return out


def pin_lse_brute_force(impl):
    lse = _lse_impl(impl)
    for (q, k, v, mask, causal, scale) in _tiny_cases():
        got = lse(q, k, v, mask=mask, is_causal=causal, scale=scale)
        ref = brute_force_lse_decimal(q, k, mask, causal, scale)
        fin = np.isfinite(ref)
        assert np.array_equal(np.isfinite(got), fin)
        assert np.all(got[~fin] == -np.inf)
        np.testing.assert_allclose(got[fin], ref[fin], rtol=0, atol=1e-13)


def pin_lse_closed_forms(impl):
    lse = _lse_impl(impl)
    g = _rng(22)
    H, L, D = 2, 7, 4
    # q = 0: every admissible score is 0, so the sum has (#keys) ones
    q0, k, v = np.zeros((H, L, D)), g.standard_normal((H, L, D)), g.standard_normal((H, L, D))
    np.testing.assert_allclose(lse(q0, k, v, is_causal=True),
                               np.broadcast_to(np.log(np.arange(1, L + 1)), (H, L)),
                               rtol=0, atol=1e-14)
    # one admissible key j: the sum is the single term exp(scale * q_i . k_j)
    q = g.standard_normal((H, L, D))
    perm = g.permutation(L)
    mask = np.ones((L, L), dtype=bool)
    mask[np.arange(L), perm] = False
    expect = 0.5 * np.einsum("hid,hid->hi", q, k[:, perm, :])
    np.testing.assert_allclose(lse(q, k, v, mask=mask, scale=0.5), expect, rtol=0, atol=1e-14)
    # a fully removed row has an empty sum: -inf
    mask2 = np.zeros((L, L), dtype=bool)
    mask2[3] = True
    got = lse(q, k, v, mask=mask2)
    assert got[0, 3] == -np.inf and got[1, 3] == -np.inf
    assert np.all(np.isfinite(np.delete(got, 3, axis=1)))


def pin_lse_torch_logsumexp(impl):
    import torch
    lse = _lse_impl(impl)
    g = _rng(23)
    B, H, L, D = 2, 3, 19, 8
    q, k, v = (g.standard_normal((B, H, L, D)) for _ in range(3))
    mask = g.random((L, L)) < 0.3
    mask[:, 0] = False
    scores = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * 0.7
    scores = scores.masked_fill(torch.from_numpy(mask), float("-inf"))
    np.testing.assert_allclose(lse(q, k, v, mask=mask, scale=0.7),
                               torch.logsumexp(scores, dim=-1).numpy(), rtol=0, atol=1e-12)


ALL_PINS = [pin_brute_force, pin_causal_row0, pin_zero_query_prefix_mean, pin_zero_scale_mean,
            pin_single_key, pin_equal_keys, pin_fully_masked_rows_zero, pin_weights_sum_to_one,
            pin_linearity_in_v, pin_permutation_invariance, pin_key_shift_invariance,
            pin_torch_math_backend, pin_lse_brute_force, pin_lse_closed_forms,
            pin_lse_torch_logsumexp]

# Pins that do not lean on a library: the mutation test requires that each
# planted mistake is caught by at least one of these alone.
INDEPENDENT_PINS = [p for p in ALL_PINS
                    if p not in (pin_torch_math_backend, pin_lse_torch_logsumexp)]

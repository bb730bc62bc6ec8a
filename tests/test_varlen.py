"""Packed variable-length documents (sdpa_forward_varlen) on the GPU: parity
with the packed-document oracle, bit-identity with the dense call on each
document's slice, untouched rows outside every document, clamped offsets.
Tolerance as in the dense parity tests: L2-relative <= 1e-2, max-abs <= 2e-2."""
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
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin), f"{what}: finite pattern differs"
    err = got[fin] - ref[fin]
    l2 = np.linalg.norm(err) / max(np.linalg.norm(ref[fin]), 1e-30)
    mx = np.abs(err).max() if err.size else 0.0
    assert l2 <= L2_TOL and mx <= MAX_TOL, f"{what}: L2-rel {l2:.3e}, max-abs {mx:.3e}"


def packed(lengths, H, D, dtype, seed):
    total = int(sum(lengths))
    q, k, v = sdpa_inputs.custom((total, H, D), dtype=dtype, seed=seed)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q, k, v, cu


def run(sdpa, q, k, v, cu, max_seqlen, causal, lse=False, out=None):
    dev = torch.device("cuda")
    qd, kd, vd = (x.to(dev) for x in (q, k, v))
    cud = torch.from_numpy(np.asarray(cu, dtype=np.int32)).to(dev)
    if out is None:
        out = torch.full_like(qd, float("nan"))
    r = sdpa.sdpa_forward_varlen(qd, kd, vd, cud, max_seqlen, out, is_causal=causal,
                                 return_lse=lse)
    rc, detail = sdpa.sdpa_last_device_status()
    assert rc == 0, f"device status bits {detail:#x}"
    return r


MIXES = [
    ([128], 2, 64, torch.bfloat16, True),
    ([1, 127, 128, 129, 300], 2, 128, torch.bfloat16, True),
    ([513, 0, 64, 1000], 3, 64, torch.float16, True),
    ([200, 77, 450], 2, 128, torch.float16, False),
    ([1000, 1, 2, 3, 255, 256, 257], 1, 64, torch.bfloat16, False),
]


@pytest.mark.parametrize("lengths,H,D,dtype,causal", MIXES,
                         ids=[f"{len(m[0])}docs-H{m[1]}-D{m[2]}-{'causal' if m[4] else 'full'}"
                              for m in MIXES])
def test_varlen_matches_oracle(sdpa_lib, lengths, H, D, dtype, causal):
    q, k, v, cu = packed(lengths, H, D, dtype, seed=900 + len(lengths) + D)
    out, lse = run(sdpa_lib, q, k, v, cu, max(lengths), causal, lse=True)
    ref, ref_lse = oracle.sdpa_varlen(q, k, v, cu, is_causal=causal, return_lse=True)
    check(out.double().cpu().numpy(), ref, "out")
    np.testing.assert_allclose(lse.double().cpu().numpy(), ref_lse, rtol=0, atol=2e-3)


def test_varlen_bitwise_equals_dense_per_document(sdpa_lib):
    lengths = [300, 1, 128, 517]
    q, k, v, cu = packed(lengths, 4, 128, torch.bfloat16, seed=930)
    out, lse = run(sdpa_lib, q, k, v, cu, max(lengths), True, lse=True)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    for a, b in zip(cu[:-1], cu[1:]):
        # the document's slice as a strided [H, len, D] view, no copy
        sl = [x[a:b].permute(1, 0, 2) for x in (qd, kd, vd)]
        o1, l1 = sdpa_lib.sdpa_forward(*sl, is_causal=True, return_lse=True)
        assert torch.equal(out[a:b].permute(1, 0, 2), o1)
        assert torch.equal(lse[:, a:b], l1)


def test_many_documents_cross_cursor_chunks(sdpa_lib):
    rng = np.random.default_rng(5)
    lengths = rng.integers(0, 200, size=300).tolist()   # 300 documents, some empty
    q, k, v, cu = packed(lengths, 2, 64, torch.bfloat16, seed=931)
    out = run(sdpa_lib, q, k, v, cu, max(lengths), True)
    ref = oracle.sdpa_varlen(q, k, v, cu, is_causal=True)
    check(out.double().cpu().numpy(), ref, "300 documents")


def test_small_max_seqlen_only_shrinks_the_grid(sdpa_lib):
    lengths = [2000, 900, 31]
    q, k, v, cu = packed(lengths, 2, 64, torch.bfloat16, seed=932)
    a = run(sdpa_lib, q, k, v, cu, max(lengths), True)
    b = run(sdpa_lib, q, k, v, cu, 1, True)   # grid of one CTA walks every unit
    assert torch.equal(a, b)


def test_rows_outside_documents_untouched(sdpa_lib):
    q, k, v = sdpa_inputs.custom((700, 2, 64), dtype=torch.bfloat16, seed=933)
    cu = np.array([100, 350, 600], dtype=np.int32)
    out = run(sdpa_lib, q, k, v, cu, 250, True)
    o = out.float().cpu()
    assert torch.isnan(o[:100]).all() and torch.isnan(o[600:]).all()
    check(out.double().cpu().numpy()[100:600],
          oracle.sdpa_varlen(q, k, v, cu, is_causal=True)[100:600], "covered rows")


def test_bad_offsets_are_clamped(sdpa_lib):
    """Offsets past the end or going backwards cannot make the kernel touch
    memory outside the buffers: each document is clamped to [0, total) with
    end >= start."""
    total = 500
    q, k, v = sdpa_inputs.custom((total, 2, 64), dtype=torch.bfloat16, seed=934)
    cu = np.array([-7, 200, 150, 420, 9999], dtype=np.int32)
    out = run(sdpa_lib, q, k, v, cu, 512, False)
    clamped = [0, 200, 200, 420, 500]        # [0,200) [200,200) [200,420) [420,500)
    check(out.double().cpu().numpy(), oracle.sdpa_varlen(q, k, v, clamped), "clamped")

"""The FMA-pipe base-2 exponential that the kernel uses for part of the
softmax probabilities (Cody-Waite range reduction plus a minimax cubic).

CPU: the constants compiled into ptx.cuh are the ones the committed fit
produces, and a float32 emulation of the kernel's operation order keeps the
relative error below 2^-13 with exact zeros for inputs at or below -127.
GPU: the device implementation (through the test entry point) meets the same
bound against the exact exponential."""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "scaled_dot_product_forward_gb300")
sys.path.insert(0, PKG)
import fit_exp2_poly as fit  # noqa: E402

REL_BOUND = 2.0 ** -13


def compiled_constants():
    text = open(os.path.join(PKG, "csrc", "ptx.cuh")).read()
    vals = {}
    for k in ("kExp2C1", "kExp2C2", "kExp2C3"):
        m = re.search(rf"constexpr float {k} = ([-+0-9.eE]+)f;", text)
        assert m, k
        vals[k] = np.float32(float(m.group(1)))
    return [np.float32(1.0), vals["kExp2C1"], vals["kExp2C2"], vals["kExp2C3"]]


def test_constants_match_fit():
    pytest.importorskip("scipy")
    fitted = fit.coefficients_f32()
    for a, b in zip(compiled_constants(), fitted):
        assert abs(float(a) - float(b)) <= 2e-7 * max(1.0, abs(float(b)))


def test_emulated_error_bound():
    c = compiled_constants()
    x = np.linspace(-126.0, 8.0, 400001).astype(np.float32)
    y = fit.exp2_poly_f32(x, c)
    rel = np.abs(y / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < REL_BOUND
    ints = np.arange(-126, 9, dtype=np.float32)
    assert np.array_equal(fit.exp2_poly_f32(ints, c), np.exp2(ints.astype(np.float64)))
    low = np.array([-127.0, -127.5, -1000.0, -np.inf], dtype=np.float32)
    assert np.array_equal(fit.exp2_poly_f32(low, c), np.zeros(4, dtype=np.float32))


@pytest.mark.gpu
def test_device_polynomial(sdpa_lib):
    import torch
    x = torch.linspace(-126.0, 8.0, 1_000_001, dtype=torch.float32)
    y = sdpa_lib.sdpa_debug_exp2_poly(x.cuda()).cpu().double()
    ref = torch.exp2(x.double())
    rel = ((y / ref) - 1.0).abs().max().item()
    assert rel < REL_BOUND, rel
    ints = torch.arange(-126, 9, dtype=torch.float32)
    assert torch.equal(sdpa_lib.sdpa_debug_exp2_poly(ints.cuda()).cpu(), torch.exp2(ints))
    low = torch.tensor([-127.0, -127.5, -1000.0, float("-inf"), -3.0e38], dtype=torch.float32)
    assert torch.equal(sdpa_lib.sdpa_debug_exp2_poly(low.cuda()).cpu(), torch.zeros(5))
    # odd length exercises the single-element tail
    odd = torch.tensor([0.5, -2.25, 3.0], dtype=torch.float32)
    got = sdpa_lib.sdpa_debug_exp2_poly(odd.cuda()).cpu().double()
    assert ((got / torch.exp2(odd.double())) - 1.0).abs().max().item() < REL_BOUND

"""The fp64 oracle against its pins (CPU only).  See ``oracle_pins.py`` for
what each pin rests on."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.sdpa)


def test_rank3_equals_rank4():
    g = np.random.default_rng(3)
    q, k, v = (g.standard_normal((3, 10, 4)) for _ in range(3))
    assert np.array_equal(oracle.sdpa(q, k, v, is_causal=True),
                          oracle.sdpa(q[None], k[None], v[None], is_causal=True)[0])


def test_causal_equals_triangular_mask():
    """is_causal and an explicit strict-upper-triangle mask are the same set of
    removed keys: query i sees j <= i."""
    g = np.random.default_rng(4)
    L = 11
    q, k, v = (g.standard_normal((2, L, 4)) for _ in range(3))
    tri = np.triu(np.ones((L, L), dtype=bool), k=1)
    assert np.array_equal(oracle.sdpa(q, k, v, is_causal=True), oracle.sdpa(q, k, v, mask=tri))


def test_rows_match_full():
    g = np.random.default_rng(5)
    B, H, L, D = 2, 3, 33, 8
    q, k, v = (g.standard_normal((B, H, L, D)) for _ in range(3))
    mask = g.random((L, L)) < 0.3
    full = oracle.sdpa(q, k, v, mask=mask)
    rows = np.array([[0, 0, 0], [1, 2, 32], [0, 1, 17], [1, 0, 5]])
    got = oracle.sdpa_rows(q, k, v, rows, mask=mask)
    assert np.array_equal(got, full[rows[:, 0], rows[:, 1], rows[:, 2]])


def test_rows_reject_out_of_range():
    q = np.zeros((1, 1, 4, 4))
    with pytest.raises(RuntimeError):
        oracle.sdpa_rows(q, q, q, [[0, 0, 4]])


def test_default_scale_is_inverse_sqrt_d():
    g = np.random.default_rng(6)
    q, k, v = (g.standard_normal((1, 5, 16)) for _ in range(3))
    assert np.array_equal(oracle.sdpa(q, k, v, is_causal=True),
                          oracle.sdpa(q, k, v, is_causal=True, scale=0.25))


def test_golden_regression_fixture():
    """Stored outputs written by tests/golden/make_oracle_fixture.py (which
    calls only the oracle); guards against accidental changes to it."""
    import json, os
    import sdpa_inputs
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small.json")
    with open(path) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        q, k, v = sdpa_inputs.custom(case["shape"], dtype=getattr(__import__("torch"), case["dtype"]),
                                     seed=case["seed"], amplitude=case["amplitude"])
        mask = None
        if case["p_masked"] is not None:
            mask = sdpa_inputs.bernoulli_mask(case["shape"][-2], case["p_masked"], case["seed"] + 3,
                                              case["n_full_rows"])
        out = oracle.sdpa(q, k, v, mask=mask, is_causal=case["is_causal"])
        flat = out.reshape(-1)
        idx = np.array(case["probe_index"])
        np.testing.assert_allclose(flat[idx], np.array(case["probe_value"]), rtol=0, atol=1e-15)
        assert abs(float(np.sum(out)) - case["sum"]) < 1e-9

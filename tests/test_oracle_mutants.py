"""Each planted mistake in a copy of the oracle source must be caught by the
independent pins (brute force, closed forms, invariants) -- without the torch
cross-check.  This shows the pins constrain every step of the definition:
the product q.k, the scale, the removal of keys, the softmax and the value
mix.  The mutants are built in a temporary directory and never replace the
real oracle."""
import functools
import os

import pytest

import oracle
from tests import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sdpa_oracle.c")

MUTANTS = {
    "causal_off_by_one": ("if (is_causal && j > i)", "if (is_causal && j >= i)"),
    "exp_sign_flipped": ("s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);"),
    "scale_dropped": ("s[j] = s[j] * scale;", "s[j] = s[j];"),
    "scale_squared": ("s[j] = s[j] * scale;", "s[j] = s[j] * scale * scale;"),
    "k_transposed": ("acc += qi[d] * kj[d];", "acc += qi[d] * K[d * L + j];"),
    "mask_polarity": ("mask_row[j] != 0", "mask_row[j] == 0"),
    "no_normalisation": ("s[j] = s[j] / total;", "s[j] = s[j];"),
    "unsafe_softmax": ("if (m == -INFINITY) {", "if (0) {"),
    "v_wrong_row": ("const double *vj = V + j * D;", "const double *vj = V + i * D;"),
    "wrong_normaliser": ("total += s[j];", "total += s[j] * s[j];"),
    "lse_without_max": ("*lse = m + log(total);", "*lse = log(total);"),
    "lse_of_empty_row_zero": ("*lse = -INFINITY; /* log of an empty sum */", "*lse = 0.0;"),
    "mask_row_of_query_0": ("mask ? mask + i * L : NULL, is_causal, scale, s,\n                               out + r * D",
                            "mask ? mask : NULL, is_causal, scale, s,\n                               out + r * D"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.load_variant(oracle.compile_source(str(mpath), str(tmp_path / "libmutant.so")))
    impl = functools.partial(oracle.sdpa, _lib_override=lib)
    caught = []
    for pin in pins.INDEPENDENT_PINS:
        try:
            pin(impl)
        except (AssertionError, RuntimeError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every independent pin"

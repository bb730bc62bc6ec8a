"""Writes oracle_small.json: outputs of the fp64 oracle (and nothing else) on
small seeded inputs from sdpa_inputs.  A regression fixture: it records what
the pinned oracle computes so that an accidental change to the oracle shows.
Run from the repository root:  python tests/golden/make_oracle_fixture.py"""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)
import oracle  # noqa: E402
import sdpa_inputs  # noqa: E402

CASES = [
    dict(shape=[4, 128, 64], dtype="bfloat16", seed=1000, amplitude=1.0, is_causal=True,
         p_masked=None, n_full_rows=0),
    dict(shape=[1, 2, 200, 128], dtype="bfloat16", seed=77, amplitude=0.5, is_causal=True,
         p_masked=None, n_full_rows=0),
    dict(shape=[1, 2, 130, 64], dtype="float16", seed=4000, amplitude=1.0, is_causal=False,
         p_masked=0.3, n_full_rows=4),
]


def main():
    out_cases = []
    for c in CASES:
        q, k, v = sdpa_inputs.custom(c["shape"], dtype=getattr(torch, c["dtype"]), seed=c["seed"],
                                     amplitude=c["amplitude"])
        mask = None
        if c["p_masked"] is not None:
            mask = sdpa_inputs.bernoulli_mask(c["shape"][-2], c["p_masked"], c["seed"] + 3,
                                              c["n_full_rows"])
        out = oracle.sdpa(q, k, v, mask=mask, is_causal=c["is_causal"])
        flat = out.reshape(-1)
        idx = np.random.default_rng(c["seed"]).choice(flat.size, size=16, replace=False)
        out_cases.append(dict(c, probe_index=[int(i) for i in idx],
                              probe_value=[float(flat[i]) for i in idx], sum=float(np.sum(out))))
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_small.json")
    with open(path, "w") as f:
        json.dump({"written_by": "tests/golden/make_oracle_fixture.py (oracle only)",
                   "cases": out_cases}, f, indent=1)
    print(path)


if __name__ == "__main__":
    main()

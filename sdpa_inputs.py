"""Seeded synthetic inputs for scaled dot-product attention.

This module is shared by the tests, the smoke check and the benchmark.  It
holds no attention arithmetic: it only draws numbers.  Both the CUDA path and
the CPU oracle consume exactly the tensors it returns (already rounded to the
16-bit input type), so any disagreement between them comes from the
computation, never from the inputs.

Recipe (one torch CPU ``Generator`` per tensor):
  seed = 1000 * workload_id + {q: 0, k: 1, v: 2, mask: 3, fully-masked rows: 4}
  q, k, v: fp32 ``randn`` times ``amplitude``, rounded to nearest-even into the
           16-bit type.
  mask:    ``rand < p_masked`` (True / 1 = key removed), then the first
           ``n_full_rows`` entries of a seeded ``randperm(L)`` become fully
           removed rows.

The profiling pages never state their shapes, so the workloads below are the
five shapes this library is specified and measured on; their distributions
(i.i.d. normal, optional 0.5 amplitude, Bernoulli(0.3) mask with 16 fully
removed rows) follow that specification.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    wid: int                 # workload number, also the seed base
    name: str
    B: int | None            # None -> rank-3 [H, L, D]
    H: int
    L: int
    D: int
    dtype: torch.dtype
    amplitude: float = 1.0
    is_causal: bool = True
    p_masked: float | None = None   # None -> no explicit mask
    n_full_rows: int = 0

    @property
    def rank(self) -> int:
        return 3 if self.B is None else 4

    @property
    def shape(self) -> tuple:
        return (self.H, self.L, self.D) if self.B is None else (self.B, self.H, self.L, self.D)

    @property
    def heads(self) -> int:
        return (1 if self.B is None else self.B) * self.H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def flops(self) -> float:
        """Algorithmic FLOPs: causal 2*B*H*L^2*D (half the score matrix);
        with an explicit mask every tile is computed, 4*B*H*L^2*D."""
        f = 2.0 * self.heads * self.L * self.L * self.D
        return f if self.is_causal else 2.0 * f

    def alg_bytes(self) -> int:
        """Read q, k, v once and write out once (+ the [L, L] mask bytes)."""
        esz = 2
        b = 4 * self.heads * self.L * self.D * esz
        if self.p_masked is not None:
            b += self.L * self.L
        return b


WORKLOADS = {
    1: Workload(1, "causal rank-3 [H=4, L=128, D=64] bf16", None, 4, 128, 64, torch.bfloat16),
    2: Workload(2, "causal [B=8, H=16, L=1024, D=64] bf16 (also as rank-3 [128, 1024, 64])",
                8, 16, 1024, 64, torch.bfloat16),
    3: Workload(3, "causal [B=4, H=32, L=4096, D=128] bf16, N(0,1)*0.5",
                4, 32, 4096, 128, torch.bfloat16, amplitude=0.5),
    4: Workload(4, "masked [B=2, H=16, L=2048, D=64] fp16, Bernoulli(0.3) mask, 16 fully masked rows",
                2, 16, 2048, 64, torch.float16, is_causal=False, p_masked=0.3, n_full_rows=16),
    5: Workload(5, "long-context causal [B=1, H=32, L=16384, D=128] bf16, N(0,1)*0.5",
                1, 32, 16384, 128, torch.bfloat16, amplitude=0.5),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal(shape, dtype, seed: int, amplitude: float = 1.0) -> torch.Tensor:
    """fp32 N(0,1) * amplitude from ``seed``, rounded into ``dtype`` (CPU)."""
    x = torch.randn(tuple(shape), generator=_gen(seed), dtype=torch.float32)
    if amplitude != 1.0:
        x = x * amplitude
    return x.to(dtype)


def bernoulli_mask(L: int, p_masked: float, seed: int, n_full_rows: int = 0,
                   rows_seed: int | None = None) -> torch.Tensor:
    """[L, L] uint8 mask, 1 = removed, with ``n_full_rows`` fully removed rows."""
    m = (torch.rand((L, L), generator=_gen(seed)) < p_masked).to(torch.uint8)
    if n_full_rows:
        perm = torch.randperm(L, generator=_gen(seed + 1 if rows_seed is None else rows_seed))
        m[perm[:n_full_rows]] = 1
    return m


def full_rows(w: Workload) -> torch.Tensor:
    """Indices of the fully removed rows of workload ``w`` (empty if none)."""
    if w.p_masked is None or w.n_full_rows == 0:
        return torch.empty(0, dtype=torch.int64)
    perm = torch.randperm(w.L, generator=_gen(1000 * w.wid + 4))
    return perm[: w.n_full_rows].sort().values


def make(w: Workload | int):
    """(q, k, v, mask) on the CPU for workload ``w``; mask is None when the
    workload has none."""
    if isinstance(w, int):
        w = WORKLOADS[w]
    base = 1000 * w.wid
    q = normal(w.shape, w.dtype, base + 0, w.amplitude)
    k = normal(w.shape, w.dtype, base + 1, w.amplitude)
    v = normal(w.shape, w.dtype, base + 2, w.amplitude)
    mask = None
    if w.p_masked is not None:
        mask = bernoulli_mask(w.L, w.p_masked, base + 3, w.n_full_rows, rows_seed=base + 4)
    return q, k, v, mask


def custom(shape, dtype=torch.bfloat16, seed: int = 0, amplitude: float = 1.0):
    """(q, k, v) of any shape from one base seed (seed, seed+1, seed+2)."""
    return (normal(shape, dtype, seed, amplitude), normal(shape, dtype, seed + 1, amplitude),
            normal(shape, dtype, seed + 2, amplitude))


def sample_rows(B: int, H: int, L: int, n: int, seed: int) -> torch.Tensor:
    """n (b, h, i) triples for sampled checks: the first and last rows of the
    first and last heads, rows around every 128-row tile edge of head 0, and
    the rest uniform at random.  Returns int64 [n', 3] with n' >= n possible
    duplicates removed."""
    g = _gen(seed)
    picks = []
    for b in {0, B - 1}:
        for h in {0, H - 1}:
            for i in {0, 1, L // 2, L - 2, L - 1}:
                if 0 <= i < L:
                    picks.append((b, h, i))
    for t in range(0, L, 128):
        for i in (t - 1, t, t + 127):
            if 0 <= i < L:
                picks.append((0, 0, i))
    while len(picks) < n:
        b = int(torch.randint(0, B, (1,), generator=g))
        h = int(torch.randint(0, H, (1,), generator=g))
        i = int(torch.randint(0, L, (1,), generator=g))
        picks.append((b, h, i))
    uniq = sorted(set(picks))
    return torch.tensor(uniq, dtype=torch.int64)


# ---------------------------------------------------------------- packed documents
VARLEN_DOCS = dict(n_docs=16, lo=512, hi=4096, step=64, H=32, D=128, seed=6000)


def varlen_lengths(n_docs: int, lo: int, hi: int, step: int, seed: int) -> list[int]:
    """Document lengths drawn uniformly from {lo, lo + step, ..., hi}."""
    g = _gen(seed)
    k = torch.randint(0, (hi - lo) // step + 1, (n_docs,), generator=g)
    return [lo + step * int(x) for x in k]


def make_varlen(n_docs=16, lo=512, hi=4096, step=64, H=32, D=128, seed=6000,
                dtype=torch.bfloat16, amplitude=0.5):
    """Packed [total, H, D] q, k, v of seeded lengths and their int32 offsets."""
    lengths = varlen_lengths(n_docs, lo, hi, step, seed)
    total = sum(lengths)
    q = normal((total, H, D), dtype, seed + 1, amplitude)
    k = normal((total, H, D), dtype, seed + 2, amplitude)
    v = normal((total, H, D), dtype, seed + 3, amplitude)
    cu = torch.zeros(n_docs + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(lengths), 0).to(torch.int32)
    return q, k, v, cu, lengths


# ---------------------------------------------------------------- sparse top-k
SPARSE_DSA = dict(total=8192, H=64, D=128, topk=2048, seed=7000)


def causal_topk_indices(total: int, topk: int, seed: int):
    """Hole-free index rows of one causal document: row i lists min(i + 1,
    topk) distinct key rows <= i in random order, then -1; and the counts."""
    g = _gen(seed)
    idx = torch.full((total, topk), -1, dtype=torch.int32)
    length = torch.empty(total, dtype=torch.int32)
    for i in range(total):
        n = min(i + 1, topk)
        if i + 1 <= topk:
            rows = torch.randperm(i + 1, generator=g)
        else:
            rows = torch.randperm(i + 1, generator=g)[:topk]
        idx[i, :n] = rows.to(torch.int32)
        length[i] = n
    return idx, length


def make_sparse(total=8192, H=64, D=128, topk=2048, seed=7000, dtype=torch.bfloat16,
                amplitude=0.5):
    """q [total, H, D]; one kv tensor [total, D] serving as the shared key and
    value head (``fwd(q, kv, idx, ...)``); causal top-k index rows and their
    counts."""
    q = normal((total, H, D), dtype, seed + 1, amplitude)
    kv = normal((total, D), dtype, seed + 2, amplitude)
    idx, length = causal_topk_indices(total, topk, seed + 4)
    return q, kv, idx, length

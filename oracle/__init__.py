"""fp64 CPU oracle for scaled dot-product attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package.  The CUDA library never loads it, and it
never loads the CUDA library.

The arithmetic lives in ``sdpa_oracle.c`` (plain C, fp64, one query row at a
time, OpenMP over rows); this module only compiles it with gcc and marshals
arrays.  It computes the five steps printed in "Profiling attention in PyTorch:
kernels, backends and where the time goes" (news.bpdata.com), section "Naiv
causal attention", and in "PyTorch attention profiling: Flash, cuDNN and Math
backends compared" (dev.smart-guide.co.kr), section 1: matmul(q, k^T), times
scale, masked_fill(mask, -inf), softmax over keys, matmul(attn, v) -- with the
math backend's safe softmax (a fully removed row gives zeros) from the
math-backend sections of the same pages.

Parity pins (see ``tests/test_oracle.py``): exact-decimal brute force on tiny
shapes, closed forms (causal row 0 -> v[0]; q = 0 -> prefix mean; one allowed
key -> that value row; equal keys -> mean of allowed values), invariants
(weights sum to one, linearity in v, key/value permutation and key-shift
invariance, zero rows for fully removed queries) and torch's CPU math backend
in fp64.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdpa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_sdpa.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, lib_path: str) -> str:
    """gcc -O2, OpenMP, no fast-math (fp64 rounding follows the source order)."""
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False) -> str:
    """Compile ``sdpa_oracle.c`` into ``liboracle_sdpa.so`` beside it."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    return compile_source(_SRC, _LIB)


def load_variant(lib_path: str):
    """Bind another build of the oracle source (the tests use this to show
    that deliberately broken copies fail the pins)."""
    return _bind(ctypes.CDLL(lib_path))


def _bind(lib):
    d, i64, u8p = ctypes.POINTER(ctypes.c_double), ctypes.c_int64, ctypes.c_void_p
    lib.oracle_sdpa_fp64.argtypes = [d, d, d, d, i64, i64, i64, i64, u8p,
                                     ctypes.c_int, ctypes.c_double, d]
    lib.oracle_sdpa_fp64.restype = ctypes.c_int
    lib.oracle_sdpa_rows_fp64.argtypes = [d, d, d, i64, i64, i64, i64, u8p,
                                          ctypes.c_int, ctypes.c_double,
                                          ctypes.POINTER(ctypes.c_int64), i64, d, d]
    lib.oracle_sdpa_rows_fp64.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs on (``OMP_NUM_THREADS`` caps it)."""
    return int(_load().oracle_num_threads())


def _as_f64(x) -> np.ndarray:
    """Widen a torch tensor or array exactly to a dense float64 numpy array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().to("cpu", torch.float64).contiguous().numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _as_mask(mask, L):
    if mask is None:
        return None
    try:
        import torch
        if isinstance(mask, torch.Tensor):
            mask = mask.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    m = np.ascontiguousarray(np.asarray(mask) != 0, dtype=np.uint8)
    if m.shape != (L, L):
        raise ValueError(f"mask must be [L, L] = [{L}, {L}], got {m.shape}")
    return m


def _shape4(q):
    if q.ndim == 3:
        return (1,) + q.shape
    if q.ndim == 4:
        return q.shape
    raise ValueError(f"q must be rank 3 [H, L, D] or rank 4 [B, H, L, D], got {q.shape}")


def default_scale(D: int) -> float:
    """1/sqrt(head_dim): the scale the NaiveCausalAttention module sets in its
    constructor on both profiling pages."""
    return 1.0 / math.sqrt(D)


def sdpa(q, k, v, mask=None, is_causal=False, scale=None, _lib_override=None,
         return_lse=False):
    """Full attention output in fp64, same rank as ``q`` ([H,L,D] or [B,H,L,D]).

    ``mask``: optional [L, L], nonzero = removed (masked_fill polarity).
    ``scale``: None -> 1/sqrt(D).  ``return_lse``: also return the per-row
    log-sum-exp of the scaled, masked scores (shape of ``q`` without D)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    if not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must share one shape")
    B, H, L, D = _shape4(q)
    m = _as_mask(mask, L)
    s = default_scale(D) if scale is None else float(scale)
    out = np.empty_like(q)
    lse = np.empty(q.shape[:-1], dtype=np.float64) if return_lse else None
    dp = ctypes.POINTER(ctypes.c_double)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_sdpa_fp64(
        q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp),
        out.ctypes.data_as(dp), B, H, L, D,
        None if m is None else m.ctypes.data, int(bool(is_causal)), s,
        None if lse is None else lse.ctypes.data_as(dp))
    if rc != 0:
        raise RuntimeError("oracle_sdpa_fp64 failed")
    return (out, lse) if return_lse else out


def sdpa_rows(q, k, v, rows, mask=None, is_causal=False, scale=None,
              _lib_override=None, return_lse=False):
    """Output rows for the (b, h, i) triples in ``rows`` (shape [n, 3]); for
    rank-3 inputs pass b = 0.  Returns [n, D] fp64 (and [n] log-sum-exp
    values with ``return_lse``)."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    B, H, L, D = _shape4(q)
    m = _as_mask(mask, L)
    idx = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    s = default_scale(D) if scale is None else float(scale)
    out = np.empty((idx.shape[0], D), dtype=np.float64)
    lse = np.empty(idx.shape[0], dtype=np.float64) if return_lse else None
    dp = ctypes.POINTER(ctypes.c_double)
    lib = _lib_override if _lib_override is not None else _load()
    rc = lib.oracle_sdpa_rows_fp64(
        q.ctypes.data_as(dp), k.ctypes.data_as(dp), v.ctypes.data_as(dp),
        B, H, L, D, None if m is None else m.ctypes.data, int(bool(is_causal)), s,
        idx.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), idx.shape[0],
        out.ctypes.data_as(dp), None if lse is None else lse.ctypes.data_as(dp))
    if rc != 0:
        raise RuntimeError("oracle_sdpa_rows_fp64 failed (row index out of range?)")
    return (out, lse) if return_lse else out


def sdpa_varlen(q, k, v, cu_seqlens, is_causal=False, scale=None, return_lse=False):
    """Packed documents: ``q, k, v`` are [total, H, D] with document i in rows
    ``[cu_seqlens[i], cu_seqlens[i+1])``, as the varlen kernels on the
    FlashInfer pull-request page ("FlashInfer, Cake DSA kernel optimization",
    blog.secrett2633.cloud, section 3) describe their per-document rows with
    cumulative offsets.  Each document is attended on its own (the attention
    above, applied to its slice); rows outside every document stay NaN.
    Returns [total, H, D] fp64 (and the log-sum-exp [H, total])."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    if q.ndim != 3 or not (q.shape == k.shape == v.shape):
        raise ValueError("q, k, v must share one [total, H, D] shape")
    cu = np.asarray(cu_seqlens, dtype=np.int64).reshape(-1)
    total, H, D = q.shape
    if cu.size < 2 or cu[0] < 0 or cu[-1] > total or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must be nondecreasing within [0, total]")
    out = np.full(q.shape, np.nan)
    lse = np.full((H, total), np.nan) if return_lse else None
    for a, b in zip(cu[:-1], cu[1:]):
        if b == a:
            continue
        sl = slice(int(a), int(b))
        # [len, H, D] -> [H, len, D]
        qs, ks, vs = (np.ascontiguousarray(x[sl].transpose(1, 0, 2)) for x in (q, k, v))
        r = sdpa(qs, ks, vs, is_causal=is_causal, scale=scale, return_lse=return_lse)
        if return_lse:
            o, l = r
            lse[:, sl] = l
        else:
            o = r
        out[sl] = o.transpose(1, 0, 2)
    return (out, lse) if return_lse else out


def sparse_compact_indices(idx_local, cu_seqlens_q, cu_seqlens_k, is_causal=True):
    """Index preparation of the sparse top-k path: per-document key positions
    (``idx_local`` [total_q, topk] int, -1 = hole) become global key rows with
    the holes removed, as the FlashInfer pull-request page ("FlashInfer,
    Cake DSA kernel optimization", blog.secrett2633.cloud) describes in its
    sections 1 and 3: each row keeps its valid entries in their order,
    rebased by the document's key offset, followed by -1; ``topk_length``
    counts them.  An entry is valid when 0 <= l < the document's key count
    and, with ``is_causal``, l <= the query's position in its document.
    Plain loops (the definition); returns (idx_global, topk_length) int64."""
    idx_local = np.asarray(idx_local, dtype=np.int64)
    cu_q = np.asarray(cu_seqlens_q, dtype=np.int64).reshape(-1)
    cu_k = np.asarray(cu_seqlens_k, dtype=np.int64).reshape(-1)
    total_q, topk = idx_local.shape
    out = np.full((total_q, topk), -1, dtype=np.int64)
    length = np.zeros(total_q, dtype=np.int64)
    for b in range(len(cu_q) - 1):
        nk = cu_k[b + 1] - cu_k[b]
        for i in range(cu_q[b], cu_q[b + 1]):
            pos = i - cu_q[b]
            n = 0
            for t in range(topk):
                l = idx_local[i, t]
                if l < 0 or l >= nk or (is_causal and l > pos):
                    continue
                out[i, n] = cu_k[b] + l
                n += 1
            length[i] = n
    return out, length


def mask_tiles(mask, tile=128):
    """Tile summary of an explicit [L, L] mask (nonzero = removed, the
    masked_fill polarity of the naive module in "Profiling attention in
    PyTorch: kernels, backends and where the time goes", news.bpdata.com):
    the mask-tile skip bitmap of the per-shape tuning row.  For each tile
    (qt, kt) of tile x tile entries: ``bits[qt, kt, r, w]`` (uint32) has bit c
    set when key kt*tile + 32w + c is removed for query qt*tile + r, with
    keys and rows outside [0, L) counted as removed; ``classes[qt, kt]`` is 0
    when no entry inside [L, L] is removed, 2 when all are, else 1.  Plain
    loops over the definition; returns (bits, classes)."""
    m = np.asarray(mask)
    L = m.shape[0]
    assert m.shape == (L, L) and tile % 32 == 0
    n = (L + tile - 1) // tile
    bits = np.zeros((n, n, tile, tile // 32), dtype=np.uint32)
    classes = np.zeros((n, n), dtype=np.uint8)
    for qt in range(n):
        for kt in range(n):
            seen_removed = seen_kept = False
            for r in range(tile):
                i = qt * tile + r
                for c in range(tile):
                    j = kt * tile + c
                    inside = i < L and j < L
                    removed = (not inside) or m[i, j] != 0
                    if removed:
                        bits[qt, kt, r, c // 32] |= np.uint32(1 << (c % 32))
                    if inside:
                        seen_removed = seen_removed or removed
                        seen_kept = seen_kept or not removed
            classes[qt, kt] = 0 if not seen_removed else (2 if not seen_kept else 1)
    return bits, classes


def sdpa_sparse(q, k, v, idx, topk_length=None, scale=None, return_lse=False):
    """Sparse top-k attention, fp64: query row ``i`` (all of its heads)
    attends to the key rows ``idx[i, :topk_length[i]]`` of one shared key /
    value head, the DeepSeek sparse attention forward of the FlashInfer
    pull-request page (``out, lse = fwd(q, kv, idx, topk_length=...)``).
    q: [total_q, H, D]; k, v: [total_k, D]; idx: [total_q, topk] global rows;
    topk_length: [total_q] (None: every entry).  A row with no key gives
    zeros and lse = -inf, as the dense path's safe softmax.  Returns
    [total_q, H, D] (and lse [total_q, H])."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    idx = np.asarray(idx, dtype=np.int64)
    total_q, H, D = q.shape
    n = np.full(total_q, idx.shape[1]) if topk_length is None else \
        np.asarray(topk_length, dtype=np.int64).reshape(-1)
    s = default_scale(D) if scale is None else float(scale)
    out = np.zeros((total_q, H, D))
    lse = np.full((total_q, H), -np.inf)
    for i in range(total_q):
        rows = idx[i, :n[i]]
        if rows.size == 0:
            continue
        ks, vs = k[rows], v[rows]                 # gathered keys and values
        sc = s * (q[i] @ ks.T)                    # [H, n]
        m = sc.max(axis=1, keepdims=True)
        e = np.exp(sc - m)
        tot = e.sum(axis=1, keepdims=True)
        out[i] = (e / tot) @ vs
        lse[i] = (m + np.log(tot))[:, 0]
    return (out, lse) if return_lse else out

"""GB300 (sm_103a) fused scaled dot-product attention forward.

A thin ctypes binding over the C ABI declared in ``include/sdpa.h``: the
Python functions carry the C names and only marshal arguments (pointers,
shapes, strides, the current stream).  Every step of the computation runs in
the CUDA kernel of ``libsdpa_gb300.so``; there is no Python or CPU fallback,
and importing this package fails loudly when the library is missing.

    out = sdpa_forward(q, k, v, is_causal=True)          # torch tensors on cuda
    out = sdpa_forward(q, k, v, mask=m)                  # m: [L, L], 1 = masked out
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

__all__ = ["sdpa_forward", "sdpa_forward_raw", "sdpa_status_string", "sdpa_last_device_status",
           "sdpa_version", "SdpaError", "load_library", "LIB_PATH", "STATUS",
           "sdpa_debug_set_wait_limit_ns", "sdpa_debug_withhold_q_load",
           "sdpa_forward_varlen", "sdpa_sparse_forward", "sdpa_sparse_compact", "SdpaPlan",
           "sdpa_mask_tiles", "sdpa_forward_masked_noalloc", "head_range",
           "sdpa_forward_heads"]

LIB_PATH = _build.LIB_PATH

STATUS = {
    0: "SDPA_OK", 1: "SDPA_ERR_NULL", 2: "SDPA_ERR_RANK", 3: "SDPA_ERR_SHAPE",
    4: "SDPA_ERR_DTYPE", 5: "SDPA_ERR_LAYOUT", 6: "SDPA_ERR_ARG", 7: "SDPA_ERR_CUDA",
    8: "SDPA_ERR_DEVICE_TIMEOUT", 9: "SDPA_ERR_DEVICE",
}
SDPA_BF16, SDPA_FP16 = 0, 1


class SdpaError(RuntimeError):
    def __init__(self, status: int, where: str = "sdpa_forward"):
        self.status = int(status)
        super().__init__(f"{where}: {sdpa_status_string(status)} (status {status})")


_lib = None


def load_library(path: str | None = None):
    """Load the shared library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(
            f"{p} is missing: build it with scaled_dot_product_forward_gb300._build.build() "
            "(the CUDA path is the only path; there is no fallback)")
    lib = ctypes.CDLL(p)
    i64p, vp = ctypes.POINTER(ctypes.c_int64), ctypes.c_void_p
    lib.sdpa_forward.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, i64p,
                                 i64p, i64p, i64p, i64p, ctypes.c_int, vp, ctypes.c_float, vp]
    lib.sdpa_forward.restype = ctypes.c_int
    lib.sdpa_status_string.argtypes = [ctypes.c_int]
    lib.sdpa_status_string.restype = ctypes.c_char_p
    lib.sdpa_last_device_status.argtypes = [vp]
    lib.sdpa_last_device_status.restype = ctypes.c_int
    lib.sdpa_last_device_status_detail.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.sdpa_last_device_status_detail.restype = ctypes.c_int
    lib.sdpa_version.argtypes = []
    lib.sdpa_version.restype = ctypes.c_int
    lib.sdpa_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.sdpa_debug_set_wait_limit_ns.restype = None
    lib.sdpa_debug_withhold_q_load.argtypes = [ctypes.c_int]
    lib.sdpa_debug_withhold_q_load.restype = None
    lib.sdpa_plan_create.argtypes = [ctypes.POINTER(vp), vp, vp, vp, vp, ctypes.c_int,
                                     ctypes.c_int, i64p, i64p, i64p, i64p, i64p, ctypes.c_int,
                                     vp, ctypes.c_float]
    lib.sdpa_plan_create.restype = ctypes.c_int
    lib.sdpa_plan_set_pointers.argtypes = [vp, vp, vp, vp, vp, vp]
    lib.sdpa_plan_set_pointers.restype = ctypes.c_int
    lib.sdpa_plan_launch.argtypes = [vp, vp]
    lib.sdpa_plan_launch.restype = ctypes.c_int
    lib.sdpa_plan_destroy.argtypes = [vp]
    lib.sdpa_plan_destroy.restype = None
    lib.sdpa_forward_lse.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, i64p,
                                     i64p, i64p, i64p, i64p, i64p, ctypes.c_int, vp,
                                     ctypes.c_float, vp]
    lib.sdpa_forward_lse.restype = ctypes.c_int
    lib.sdpa_plan_set_lse.argtypes = [vp, vp, i64p]
    lib.sdpa_plan_set_lse.restype = ctypes.c_int
    lib.sdpa_forward_varlen.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, i64p, i64p, i64p, i64p,
                                        i64p, vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_float, vp]
    lib.sdpa_forward_varlen.restype = ctypes.c_int
    lib.sdpa_sparse_forward.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, i64p,
                                        ctypes.c_int64, ctypes.c_int64, i64p, i64p, vp,
                                        ctypes.c_int64, ctypes.c_int64, vp, ctypes.c_float, vp]
    lib.sdpa_sparse_forward.restype = ctypes.c_int
    lib.sdpa_sparse_compact.argtypes = [vp, ctypes.c_int64, vp, ctypes.c_int64, vp,
                                        ctypes.c_int64, ctypes.c_int64, vp, vp, ctypes.c_int64,
                                        ctypes.c_int, vp]
    lib.sdpa_sparse_compact.restype = ctypes.c_int
    lib.sdpa_mask_tiles.argtypes = [vp, ctypes.c_int64, vp, vp, vp]
    lib.sdpa_mask_tiles.restype = ctypes.c_int
    lib.sdpa_forward_masked_noalloc.argtypes = [vp, vp, vp, vp, ctypes.c_int, ctypes.c_int, i64p,
                                                i64p, i64p, i64p, i64p, vp, ctypes.c_float, vp]
    lib.sdpa_forward_masked_noalloc.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def sdpa_status_string(status: int) -> str:
    return load_library().sdpa_status_string(int(status)).decode()


def sdpa_version() -> int:
    return int(load_library().sdpa_version())


def sdpa_debug_set_wait_limit_ns(ns: int) -> None:
    load_library().sdpa_debug_set_wait_limit_ns(int(ns))


def sdpa_debug_withhold_q_load(enable: bool) -> None:
    load_library().sdpa_debug_withhold_q_load(1 if enable else 0)


def _arr(vals):
    return (ctypes.c_int64 * len(vals))(*[int(x) for x in vals])


def sdpa_forward_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, dtype: int, rank: int,
                     shape, q_stride, k_stride, v_stride, o_stride, is_causal: bool,
                     mask_ptr: int | None, scale: float, stream: int) -> int:
    """Call the C ABI with plain integers (device addresses, element strides,
    a cudaStream_t handle).  Returns the status code without raising."""
    lib = load_library()
    return int(lib.sdpa_forward(
        ctypes.c_void_p(q_ptr), ctypes.c_void_p(k_ptr), ctypes.c_void_p(v_ptr),
        ctypes.c_void_p(out_ptr), int(dtype), int(rank), _arr(shape),
        _arr(q_stride), _arr(k_stride), _arr(v_stride), _arr(o_stride),
        1 if is_causal else 0, ctypes.c_void_p(mask_ptr) if mask_ptr else None,
        ctypes.c_float(scale), ctypes.c_void_p(stream) if stream else None))


def sdpa_forward(q, k, v, out=None, *, is_causal: bool = False, mask=None, scale=None,
                 stream=None, return_lse: bool = False, lse=None):
    """Fused attention forward on torch CUDA tensors.

    q, k, v: [H, L, D] or [B, H, L, D], bf16 or fp16, any strides with the
    last one 1.  mask: optional [L, L] bool/uint8 on the same device (True /
    nonzero = removed).  scale: None -> 1/sqrt(D).  out: optional
    preallocated output (may be a strided view).  Launches on ``stream`` (a
    torch.cuda.Stream) or the current stream; returns ``out``, or
    ``(out, lse)`` with ``return_lse`` (lse: fp32, q's shape without D; an
    existing buffer may be passed as ``lse``).
    """
    import torch

    if q.dtype == torch.bfloat16:
        dt = SDPA_BF16
    elif q.dtype == torch.float16:
        dt = SDPA_FP16
    else:
        raise SdpaError(4)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise SdpaError(4)
    if q.shape != k.shape or q.shape != v.shape:
        raise SdpaError(3)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    elif out.dtype != q.dtype or out.shape != q.shape:
        raise SdpaError(3)
    mptr = None
    if mask is not None:
        if mask.dtype == torch.bool:
            mask = mask.view(torch.uint8)
        if mask.dtype != torch.uint8 or not mask.is_contiguous():
            raise SdpaError(5)
        mptr = mask.data_ptr()
    s = float("nan") if scale is None else float(scale)
    st = (stream if stream is not None else torch.cuda.current_stream(q.device)).cuda_stream
    if not (return_lse or lse is not None):
        rc = sdpa_forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dt,
                              q.dim(), list(q.shape), q.stride(), k.stride(), v.stride(),
                              out.stride(), is_causal, mptr, s, st)
        if rc != 0:
            raise SdpaError(rc)
        return out
    if lse is None:
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=q.device)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != tuple(q.shape[:-1]):
        raise SdpaError(3)
    rc = load_library().sdpa_forward_lse(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()), dt, q.dim(), _arr(q.shape), _arr(q.stride()),
        _arr(k.stride()), _arr(v.stride()), _arr(out.stride()), _arr(lse.stride()),
        1 if is_causal else 0, ctypes.c_void_p(mptr) if mptr else None, ctypes.c_float(s),
        ctypes.c_void_p(st) if st else None)
    if rc != 0:
        raise SdpaError(rc, "sdpa_forward_lse")
    return out, lse


def sdpa_forward_masked_noalloc(q, k, v, mask, out, *, scale=None, stream=None) -> int:
    """Masked forward whose mask summary lives in the library's fixed device
    array (sdpa_forward_masked_noalloc): nothing is allocated, so ``out``
    must be passed.  Returns the status code without raising (the caller
    decides; SDPA_ERR_SHAPE = 3 for L beyond the array's limit)."""
    import torch

    if q.dtype not in (torch.bfloat16, torch.float16):
        return 4
    mp = _mask_ptr(mask)
    s = float("nan") if scale is None else float(scale)
    st = (stream if stream is not None else torch.cuda.current_stream(q.device)).cuda_stream
    return int(load_library().sdpa_forward_masked_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), _dtype_code(q), q.dim(),
        _arr(q.shape), _arr(q.stride()), _arr(k.stride()), _arr(v.stride()), _arr(out.stride()),
        ctypes.c_void_p(mp) if mp else None, ctypes.c_float(s),
        ctypes.c_void_p(st) if st else None))


def sdpa_forward_varlen(q, k, v, cu_seqlens, max_seqlen, out=None, *, is_causal: bool = False,
                        scale=None, stream=None, return_lse: bool = False, lse=None):
    """Packed variable-length sequences (sdpa_forward_varlen).

    q, k, v: [total, H, D] bf16/fp16 CUDA tensors (any strides with the last
    one 1); cu_seqlens: int32 CUDA tensor [n_seqs + 1] of row offsets, each
    sequence attending only to itself; max_seqlen: an upper bound on the
    lengths.  Returns ``out`` [total, H, D], or ``(out, lse)`` with lse fp32
    [H, total].
    """
    import torch

    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise SdpaError(4)
    if q.dim() != 3 or q.shape != k.shape or q.shape != v.shape:
        raise SdpaError(3)
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise SdpaError(5)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    elif out.dtype != q.dtype or out.shape != q.shape:
        raise SdpaError(3)
    want_lse = return_lse or lse is not None
    if want_lse:
        if lse is None:
            lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
        elif lse.dtype != torch.float32 or tuple(lse.shape) != (q.shape[1], q.shape[0]):
            raise SdpaError(3)
    s = float("nan") if scale is None else float(scale)
    st = (stream if stream is not None else torch.cuda.current_stream(q.device)).cuda_stream
    rc = load_library().sdpa_forward_varlen(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()) if want_lse else None, dt, q.shape[0], q.shape[1],
        q.shape[2], _arr(q.stride()), _arr(k.stride()), _arr(v.stride()), _arr(out.stride()),
        _arr(lse.stride()) if want_lse else None, ctypes.c_void_p(cu_seqlens.data_ptr()),
        cu_seqlens.numel() - 1, int(max_seqlen), 1 if is_causal else 0, ctypes.c_float(s),
        ctypes.c_void_p(st) if st else None)
    if rc != 0:
        raise SdpaError(rc, "sdpa_forward_varlen")
    return (out, lse) if want_lse else out


def sdpa_sparse_forward(q, k, v, idx, topk_length=None, out=None, *, scale=None, stream=None,
                        return_lse: bool = False, lse=None):
    """Sparse top-k attention (sdpa_sparse_forward).

    q: [total_q, H, D]; k, v: [total_k, D] (one key/value head shared by all
    query heads; pass the same tensor twice for one kv tensor); idx: int32
    [total_q, topk] global key rows; topk_length: optional int32 [total_q].
    Returns ``out`` [total_q, H, D], or ``(out, lse)`` with lse fp32
    [total_q, H]."""
    import torch

    dt = _dtype_code(q)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise SdpaError(4)
    if q.dim() != 3 or k.dim() != 2 or v.shape != k.shape or k.shape[1] != q.shape[2]:
        raise SdpaError(3)
    if k.stride(1) != 1 or v.stride(1) != 1 or q.stride(2) != 1:
        raise SdpaError(5)
    if idx.dtype != torch.int32 or idx.dim() != 2 or idx.shape[0] != q.shape[0] or idx.stride(1) != 1:
        raise SdpaError(5)
    if topk_length is not None and (topk_length.dtype != torch.int32 or
                                    not topk_length.is_contiguous() or
                                    topk_length.numel() != q.shape[0]):
        raise SdpaError(5)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    elif out.dtype != q.dtype or out.shape != q.shape:
        raise SdpaError(3)
    want_lse = return_lse or lse is not None
    if want_lse:
        if lse is None:
            lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
        elif lse.dtype != torch.float32 or tuple(lse.shape) != tuple(q.shape[:2]):
            raise SdpaError(3)
    s = float("nan") if scale is None else float(scale)
    st = (stream if stream is not None else torch.cuda.current_stream(q.device)).cuda_stream
    rc = load_library().sdpa_sparse_forward(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
        ctypes.c_void_p(lse.data_ptr()) if want_lse else None, dt, q.shape[0], k.shape[0],
        q.shape[1], q.shape[2], _arr(q.stride()[:2]), k.stride(0), v.stride(0),
        _arr(out.stride()[:2]), _arr(lse.stride()) if want_lse else None,
        ctypes.c_void_p(idx.data_ptr()), idx.stride(0), idx.shape[1],
        ctypes.c_void_p(topk_length.data_ptr()) if topk_length is not None else None,
        ctypes.c_float(s), ctypes.c_void_p(st) if st else None)
    if rc != 0:
        raise SdpaError(rc, "sdpa_sparse_forward")
    return (out, lse) if want_lse else out


def sdpa_sparse_compact(idx_local, cu_seqlens_q, cu_seqlens_k, *, is_causal: bool = True,
                        stream=None):
    """Index preparation (sdpa_sparse_compact): per-document key positions
    ``idx_local`` (int32 [total_q, topk], -1 = hole) -> (global rows with the
    holes removed and -1 after them, valid counts int32 [total_q])."""
    import torch

    for t in (idx_local, cu_seqlens_q, cu_seqlens_k):
        if t.dtype != torch.int32:
            raise SdpaError(5)
    if idx_local.dim() != 2 or idx_local.stride(1) != 1:
        raise SdpaError(5)
    if not (cu_seqlens_q.is_contiguous() and cu_seqlens_k.is_contiguous()) or \
            cu_seqlens_q.numel() != cu_seqlens_k.numel():
        raise SdpaError(3)
    total_q, topk = idx_local.shape
    idx_global = torch.empty((total_q, topk), dtype=torch.int32, device=idx_local.device)
    length = torch.empty(total_q, dtype=torch.int32, device=idx_local.device)
    st = (stream if stream is not None else torch.cuda.current_stream(idx_local.device)).cuda_stream
    rc = load_library().sdpa_sparse_compact(
        ctypes.c_void_p(idx_local.data_ptr()), idx_local.stride(0),
        ctypes.c_void_p(idx_global.data_ptr()), idx_global.stride(0),
        ctypes.c_void_p(length.data_ptr()), total_q, topk,
        ctypes.c_void_p(cu_seqlens_q.data_ptr()), ctypes.c_void_p(cu_seqlens_k.data_ptr()),
        cu_seqlens_q.numel() - 1, 1 if is_causal else 0, ctypes.c_void_p(st) if st else None)
    if rc != 0:
        raise SdpaError(rc, "sdpa_sparse_compact")
    return idx_global, length


def sdpa_mask_tiles(mask, *, stream=None):
    """Mask summary (sdpa_mask_tiles) of a device [L, L] bool/uint8 mask
    (nonzero = removed): (bits int32 [n, n, 128, 4], classes uint8 [n, n])
    for n = ceil(L / 128) tiles of 128 x 128; bits[qt, kt, r, w] bit c = key
    kt*128 + 32w + c removed for row qt*128 + r (past L: removed); class 0 =
    the tile removes no entry inside [L, L], 1 = some, 2 = all."""
    import torch

    if mask.dim() != 2 or mask.shape[0] != mask.shape[1] or not mask.is_contiguous():
        raise SdpaError(3)
    if mask.dtype not in (torch.bool, torch.uint8):
        raise SdpaError(4)
    L = mask.shape[0]
    n = (L + 127) // 128
    bits = torch.empty((n, n, 128, 4), dtype=torch.int32, device=mask.device)
    classes = torch.empty((n, n), dtype=torch.uint8, device=mask.device)
    st = (stream if stream is not None else torch.cuda.current_stream(mask.device)).cuda_stream
    rc = load_library().sdpa_mask_tiles(
        ctypes.c_void_p(mask.data_ptr()), L, ctypes.c_void_p(bits.data_ptr()),
        ctypes.c_void_p(classes.data_ptr()), ctypes.c_void_p(st) if st else None)
    if rc != 0:
        raise SdpaError(rc, "sdpa_mask_tiles")
    return bits, classes


def _dtype_code(q):
    import torch
    if q.dtype == torch.bfloat16:
        return SDPA_BF16
    if q.dtype == torch.float16:
        return SDPA_FP16
    raise SdpaError(4)


def _mask_ptr(mask):
    import torch
    if mask is None:
        return None
    if mask.dtype == torch.bool:
        mask = mask.view(torch.uint8)
    if mask.dtype != torch.uint8 or not mask.is_contiguous():
        raise SdpaError(5)
    return mask.data_ptr()


class SdpaPlan:
    """A validated, pre-encoded forward (sdpa_plan_create): ``launch()`` only
    enqueues the kernel.  Bound to the shapes, strides, dtype, mask mode and
    scale given here; ``set_pointers`` moves it to other tensors of the same
    layout.  Keep the tensors alive while launches are in flight."""

    def __init__(self, q, k, v, out, *, is_causal=False, mask=None, scale=None):
        lib = load_library()
        handle = ctypes.c_void_p(None)
        s = float("nan") if scale is None else float(scale)
        rc = lib.sdpa_plan_create(
            ctypes.byref(handle), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), _dtype_code(q),
            q.dim(), _arr(q.shape), _arr(q.stride()), _arr(k.stride()), _arr(v.stride()),
            _arr(out.stride()), 1 if is_causal else 0,
            ctypes.c_void_p(_mask_ptr(mask)) if mask is not None else None, ctypes.c_float(s))
        if rc != 0:
            raise SdpaError(rc, "sdpa_plan_create")
        self._lib, self._h = lib, handle

    def set_pointers(self, q, k, v, out, mask=None):
        mp = _mask_ptr(mask)
        rc = self._lib.sdpa_plan_set_pointers(
            self._h, ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
            ctypes.c_void_p(mp) if mp else None)
        if rc != 0:
            raise SdpaError(rc, "sdpa_plan_set_pointers")

    def set_lse(self, lse=None):
        """Also write the per-row log-sum-exp into ``lse`` (fp32, q's shape
        without D) on every launch; None removes it."""
        if lse is None:
            rc = self._lib.sdpa_plan_set_lse(self._h, None, None)
        else:
            rc = self._lib.sdpa_plan_set_lse(self._h, ctypes.c_void_p(lse.data_ptr()),
                                             _arr(lse.stride()))
        if rc != 0:
            raise SdpaError(rc, "sdpa_plan_set_lse")

    def launch(self, stream=None):
        import torch
        st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
        rc = self._lib.sdpa_plan_launch(self._h, ctypes.c_void_p(st) if st else None)
        if rc != 0:
            raise SdpaError(rc, "sdpa_plan_launch")

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            self._lib.sdpa_plan_destroy(self._h)
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:  # pragma: no cover - interpreter shutdown
            pass


def sdpa_last_device_status(stream=None):
    """(status, detail bits) after synchronising ``stream``
    (sdpa_last_device_status_detail; sdpa_last_device_status is the same
    query without the bits)."""
    import torch

    st = (stream if stream is not None else torch.cuda.current_stream()).cuda_stream
    detail = ctypes.c_uint32(0)
    rc = load_library().sdpa_last_device_status_detail(ctypes.c_void_p(st) if st else None,
                                                       ctypes.byref(detail))
    return int(rc), int(detail.value)


def head_range(n_heads: int, rank: int, world: int) -> tuple[int, int]:
    """Heads ``[h0, h1)`` of rank ``rank`` among ``world`` ranks: contiguous
    ranges, the first ``n_heads % world`` ranks one head more.  Every (batch,
    head) of the forward is independent, so ranks that each compute their
    range of the same problem produce the whole output between them with no
    exchange (a rank may get no head when world > n_heads)."""
    if world < 1 or not 0 <= rank < world or n_heads < 0:
        raise ValueError(f"rank {rank} of {world} ranks, {n_heads} heads")
    base, extra = divmod(n_heads, world)
    h0 = rank * base + min(rank, extra)
    return h0, h0 + base + (1 if rank < extra else 0)


def sdpa_forward_heads(q, k, v, out, h0: int, h1: int, **kw):
    """``sdpa_forward`` on heads ``[h0, h1)`` only: q, k, v and out
    ([B, H, L, D] or [H, L, D]) are narrowed to those heads as strided views,
    so the call reads and writes that range in place.  Returns ``out``."""
    hd = 1 if q.dim() == 4 else 0
    if not 0 <= h0 <= h1 <= q.shape[hd]:
        raise SdpaError(3)
    if h0 < h1:
        sdpa_forward(q.narrow(hd, h0, h1 - h0), k.narrow(hd, h0, h1 - h0),
                     v.narrow(hd, h0, h1 - h0), out.narrow(hd, h0, h1 - h0), **kw)
    return out


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)

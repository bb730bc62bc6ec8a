"""Host-side tests of the C ABI (no GPU needed): the library builds for
sm_103a, loads, exports every function the header declares, and rejects bad
arguments with the documented status codes before touching CUDA."""
import ctypes
import math
import os
import re

import pytest

from scaled_dot_product_forward_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    import scaled_dot_product_forward_gb300 as sdpa
    return sdpa


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"SDPA_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ["sdpa_forward", "sdpa_status_string", "sdpa_last_device_status", "sdpa_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    cdll = ctypes.CDLL(_build.LIB_PATH)
    for name in declared_functions():
        assert hasattr(cdll, name), f"{name} declared in sdpa.h but not exported"


def test_only_declared_symbols_are_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {s for s in exported if "sdpa" in s}
    assert ours == set(declared_functions())


def test_status_strings(lib):
    for code, name in lib.STATUS.items():
        assert lib.sdpa_status_string(code).startswith(name)
    assert lib.sdpa_status_string(99) == "SDPA_UNKNOWN_STATUS"
    assert lib.sdpa_version() == 100


# Fake, well-aligned device addresses: validation only does arithmetic on them.
# Stand-in device addresses: the argument checks reject every call below on
# the host before any CUDA call.  A call that would pass validation is made
# only where no device exists (it must then fail with SDPA_ERR_CUDA); with a
# device it would launch a kernel on these addresses.
Q, K, V, O, M = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000


def contiguous(shape):
    st, acc = [], 1
    for e in reversed(shape):
        st.append(acc)
        acc *= e
    return list(reversed(st))


def call(lib, q=Q, k=K, v=V, o=O, dtype=0, rank=4, shape=(2, 3, 256, 64), strides=None,
         causal=1, mask=None, scale=float("nan")):
    st = strides or contiguous(shape)
    return lib.sdpa_forward_raw(q, k, v, o, dtype, rank, list(shape), st, st, st, st, causal,
                                mask, scale, 0)


def test_null_pointers(lib):
    assert call(lib, q=0) == 1
    assert call(lib, o=0) == 1
    c = ctypes.CDLL(_build.LIB_PATH)
    c.sdpa_forward.restype = ctypes.c_int
    assert c.sdpa_forward(ctypes.c_void_p(Q), ctypes.c_void_p(K), ctypes.c_void_p(V),
                          ctypes.c_void_p(O), 0, 4, None, None, None, None, None, 1, None,
                          ctypes.c_float(1.0), None) == 1


def test_rank(lib):
    assert call(lib, rank=2, shape=(256, 64)) == 2
    assert call(lib, rank=5, shape=(1, 2, 3, 256, 64)) == 2


def test_dtype(lib):
    assert call(lib, dtype=2) == 4


@pytest.mark.parametrize("shape", [(2, 3, 256, 96), (2, 3, 256, 32), (2, 3, 0, 64),
                                   (0, 3, 256, 64), (65536, 65536, 256, 64)])
def test_shape(lib, shape):
    assert call(lib, shape=shape) == 3


def test_layout(lib):
    shape = (2, 3, 256, 64)
    st = contiguous(shape)
    assert call(lib, strides=st[:3] + [2]) == 5                    # inner stride != 1
    assert call(lib, strides=[st[0], st[1], 68, 1]) == 5           # row stride not 16-byte multiple
    assert call(lib, q=Q + 8) == 5                                 # pointer not 16-byte aligned
    assert call(lib, strides=[st[0], 0, st[2], 1]) == 5            # broadcast head stride
    assert call(lib, strides=[st[0], st[1], -64, 1]) == 5          # negative stride


def test_args(lib):
    assert call(lib, causal=1, mask=M) == 6                        # causal and mask together
    assert call(lib, o=Q + 512) == 6                               # out overlaps q
    assert call(lib, scale=math.inf) == 6
    L = 256
    assert call(lib, causal=0, mask=O + 2 * 2 * 3 * L * 64 - 64) == 6   # mask overlaps out


def test_lse_argument_checks(lib):
    import ctypes
    c = ctypes.CDLL(_build.LIB_PATH)
    c.sdpa_forward_lse.restype = ctypes.c_int
    shape = (2, 3, 256, 64)
    st = contiguous(shape)
    arr = lambda vals: (ctypes.c_int64 * len(vals))(*vals)
    def call_lse(lse, lse_stride):
        return c.sdpa_forward_lse(ctypes.c_void_p(Q), ctypes.c_void_p(K), ctypes.c_void_p(V),
                                  ctypes.c_void_p(O), ctypes.c_void_p(lse), 0, 4, arr(shape),
                                  arr(st), arr(st), arr(st), arr(st),
                                  arr(lse_stride) if lse_stride else None, 1, None,
                                  ctypes.c_float(float("nan")), None)
    assert call_lse(0, [768, 256, 1]) == 1                # NULL lse
    assert call_lse(M, None) == 1                          # NULL strides
    assert call_lse(M + 2, [768, 256, 1]) == 5             # not 4-byte aligned
    assert call_lse(M, [768, 0, 1]) == 5                   # zero stride on an extent > 1
    assert call_lse(O + 64, [768, 256, 1]) == 6            # overlaps out


def test_rank3_shape_accepted_by_validation(lib):
    """A rank-3 [H, L, D] call passes validation; without a GPU it then fails
    loudly with SDPA_ERR_CUDA (there is no CPU fallback)."""
    import torch
    if torch.cuda.is_available():
        # the call would pass validation and launch on the stand-in addresses
        pytest.skip("a real device is present; validation-only check")
    assert call(lib, rank=3, shape=(4, 128, 64)) == 7


def test_permuted_view_accepted_by_validation(lib):
    import torch
    # [B, L, H, D] buffer viewed as [B, H, L, D]
    B, H, L, D = 2, 3, 256, 64
    st = [L * H * D, D, H * D, 1]
    if torch.cuda.is_available():
        # the call would pass validation and launch on the stand-in addresses
        pytest.skip("a real device is present; validation-only check")
    assert call(lib, shape=(B, H, L, D), strides=st) == 7


def test_python_wrapper_type_checks(lib):
    import torch
    x = torch.zeros(1, 2, 8, 64, dtype=torch.float32)
    with pytest.raises(lib.SdpaError):
        lib.sdpa_forward(x, x, x, is_causal=True)
    y = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    z = torch.zeros(1, 2, 8, 64, dtype=torch.float16)
    with pytest.raises(lib.SdpaError):
        lib.sdpa_forward(y, z, y, is_causal=True)


def test_varlen_argument_checks(lib):
    """sdpa_forward_varlen validates on the host before any CUDA call."""
    import ctypes
    import torch
    c = ctypes.CDLL(_build.LIB_PATH)
    c.sdpa_forward_varlen.restype = ctypes.c_int
    arr = lambda vals: (ctypes.c_int64 * len(vals))(*vals)
    total, H, D = 512, 2, 64
    st = [H * D, D, 1]                       # (token, head, dim)
    CU = M                                  # any aligned address stands for the offsets

    def call_v(cu=CU, n_seqs=3, max_seqlen=256, strides=st, o=O, lse=0, lse_stride=None,
               dim=D, causal=1):
        return c.sdpa_forward_varlen(
            ctypes.c_void_p(Q), ctypes.c_void_p(K), ctypes.c_void_p(V), ctypes.c_void_p(o),
            ctypes.c_void_p(lse) if lse else None, 0, ctypes.c_int64(total), ctypes.c_int64(H),
            ctypes.c_int64(dim), arr(strides), arr(strides), arr(strides), arr(strides),
            arr(lse_stride) if lse_stride else None, ctypes.c_void_p(cu) if cu else None,
            ctypes.c_int64(n_seqs), ctypes.c_int64(max_seqlen), causal,
            ctypes.c_float(float("nan")), None)
    assert call_v(cu=0) == 1                                  # NULL offsets
    assert call_v(n_seqs=0) == 3                              # no sequence
    assert call_v(max_seqlen=0) == 3
    assert call_v(dim=96) == 3                                # head dim
    assert call_v(cu=CU + 2) == 5                             # offsets not 4-byte aligned
    assert call_v(strides=[H * D, D, 2]) == 5                 # dim stride != 1
    assert call_v(strides=[H * D + 4, D, 1]) == 5             # token stride not 16-byte multiple
    assert call_v(o=Q + 1024) == 6                            # out overlaps q
    assert call_v(cu=O + 64) == 6                             # offsets inside out
    assert call_v(lse=M + 4096, lse_stride=None) == 1         # lse without strides
    if not torch.cuda.is_available():
        # valid: fails loudly, no fallback (never made where a device would
        # launch on the stand-in addresses)
        assert call_v() == 7


def test_sparse_argument_checks(lib):
    """sdpa_sparse_forward and sdpa_sparse_compact validate on the host."""
    import ctypes
    import torch
    c = ctypes.CDLL(_build.LIB_PATH)
    c.sdpa_sparse_forward.restype = ctypes.c_int
    c.sdpa_sparse_compact.restype = ctypes.c_int
    arr = lambda vals: (ctypes.c_int64 * len(vals))(*vals)
    total_q, total_k, H, D, topk = 64, 512, 16, 128, 128
    IDX = M

    def fwd(q=Q, o=O, idx=IDX, dim=D, qs=(H * D, D), ks=D, topk_=topk, idx_st=topk, lse=0,
            lse_stride=None):
        return c.sdpa_sparse_forward(
            ctypes.c_void_p(q), ctypes.c_void_p(K), ctypes.c_void_p(V), ctypes.c_void_p(o),
            ctypes.c_void_p(lse) if lse else None, 0, ctypes.c_int64(total_q),
            ctypes.c_int64(total_k), ctypes.c_int64(H), ctypes.c_int64(dim), arr(qs),
            ctypes.c_int64(ks), ctypes.c_int64(D), arr((H * D, D)),
            arr(lse_stride) if lse_stride else None, ctypes.c_void_p(idx) if idx else None,
            ctypes.c_int64(idx_st), ctypes.c_int64(topk_), None, ctypes.c_float(float("nan")),
            None)
    assert fwd(idx=0) == 1                       # NULL index array
    assert fwd(lse=M + 65536) == 1               # lse without strides
    assert fwd(dim=96) == 3
    assert fwd(topk_=0) == 3
    assert fwd(q=Q + 8) == 5                     # q not 16-byte aligned
    assert fwd(qs=(H * D + 4, D)) == 5           # token stride not a multiple of 8
    assert fwd(ks=D + 2) == 5
    assert fwd(idx=IDX + 2) == 5                 # index array not 4-byte aligned
    assert fwd(idx_st=topk - 1) == 5
    assert fwd(o=Q + 256) == 6                   # out overlaps q
    if not torch.cuda.is_available():
        assert fwd() == 7                        # valid: never made where a device exists

    def compact(g=O, n=O + (1 << 20), cu_q=M, cu_k=M + 4096, n_docs=2, stride_in=topk):
        return c.sdpa_sparse_compact(
            ctypes.c_void_p(IDX + (1 << 22)), ctypes.c_int64(stride_in), ctypes.c_void_p(g),
            ctypes.c_int64(topk), ctypes.c_void_p(n), ctypes.c_int64(total_q),
            ctypes.c_int64(topk), ctypes.c_void_p(cu_q) if cu_q else None, ctypes.c_void_p(cu_k),
            ctypes.c_int64(n_docs), 1, None)
    assert compact(cu_q=0) == 1
    assert compact(n_docs=0) == 3
    assert compact(stride_in=topk - 1) == 5
    assert compact(g=O + 2) == 5
    assert compact(n=O + 64) == 6                # lengths overlap the global rows

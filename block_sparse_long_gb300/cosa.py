"""Thin Python binding of libcosa's C ABI (include/cosa.h).

Argument marshalling only: every step of KAP and OSK runs in the CUDA kernels of
libcosa.so.  PyTorch supplies device memory and the current stream.  If the library is
missing the calls raise; there is no fallback.

The functions carry the C names:
  cosa_proxy_select    KAP  (CoSA Sec. 4.2, Eqs. (8)-(14))      -> mask, mask_len
  cosa_sparse_prefill  OSK  (CoSA Sec. 4.3, Algorithm A)       -> out (and visit flags)
  cosa_proxy_workspace_size, cosa_prefill_workspace_size, cosa_status_string, cosa_version
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcosa.so")

COSA_OK = 0
COSA_ERR_INVALID_ARG = -1
COSA_ERR_UNSUPPORTED = -2
COSA_ERR_CUDA = -3
COSA_ERR_DEVICE_TIMEOUT = -4
COSA_ERR_WORKSPACE = -5
COSA_ERR_BAD_INPUT = -6

VISIT_COMPUTED, VISIT_SKIPPED, VISIT_IGNORED = 0, 1, 2

# Every symbol include/cosa.h declares.
EXPORTS = ("cosa_version", "cosa_status_string", "cosa_proxy_workspace_size", "cosa_proxy_select",
           "cosa_proxy_select_static", "cosa_prefill_workspace_size", "cosa_sparse_prefill")
STATIC_SCRATCH_BYTES = 64 << 20   # COSA_STATIC_SCRATCH_BYTES


class CosaParams(ctypes.Structure):
    """Mirror of ``cosa_params``."""
    _fields_ = [
        ("num_reqs", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("stride", ctypes.c_int32), ("total_tokens", ctypes.c_int32), ("max_seqlen", ctypes.c_int32),
        ("num_pages", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32), ("mask_pitch", ctypes.c_int32),
        ("budget_ppm", ctypes.c_int32), ("flags", ctypes.c_int32), ("sm_scale", ctypes.c_double),
        ("skip_delta", ctypes.c_double),
    ]


class CosaError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {cosa_status_string(code)} ({code})")
        self.code = code


_lib = None


def library() -> ctypes.CDLL:
    """Load libcosa.so once.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m block_sparse_long_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, sz, i32p, u8p = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_void_p
    pp = ctypes.POINTER(CosaParams)
    lib.cosa_version.restype = ctypes.c_int
    lib.cosa_status_string.restype = ctypes.c_char_p
    lib.cosa_status_string.argtypes = [ctypes.c_int]
    lib.cosa_proxy_workspace_size.restype = sz
    lib.cosa_proxy_workspace_size.argtypes = [pp]
    lib.cosa_prefill_workspace_size.restype = sz
    lib.cosa_prefill_workspace_size.argtypes = [pp]
    lib.cosa_proxy_select.restype = ctypes.c_int
    lib.cosa_proxy_select.argtypes = [pp, vp, i32p, vp, i32p, i32p, i32p, vp, sz, i32p, vp]
    lib.cosa_proxy_select_static.restype = ctypes.c_int
    lib.cosa_proxy_select_static.argtypes = [pp, vp, i32p, vp, i32p, i32p, i32p, i32p, vp]
    lib.cosa_sparse_prefill.restype = ctypes.c_int
    lib.cosa_sparse_prefill.argtypes = [pp, vp, i32p, vp, vp, i32p, i32p, i32p, vp, u8p, vp, sz, i32p, vp]
    _lib = lib
    return lib


def cosa_version() -> int:
    return int(library().cosa_version())


def cosa_status_string(code: int) -> str:
    return library().cosa_status_string(int(code)).decode()


COSA_FLAG_TEST_STALL = 1   # test hook of cosa_sparse_prefill: every in-kernel wait runs out
COSA_FLAG_ASCENDING_ORDER = 2   # cosa_proxy_select writes the selected blocks in ascending order
COSA_FLAG_BINARY_MASK = 4       # cosa_sparse_prefill reads mask rows as binary block masks
COSA_FLAG_TOP_P = 8             # cosa_proxy_select: budget_ppm is the top-p threshold p
COSA_FLAG_GQA_UNION = 16        # cosa_sparse_prefill: two query heads of a kv group share one K stream
VISIT_SHARED_LOAD = 4           # visit-flag bit under COSA_FLAG_GQA_UNION: K loaded once for both heads


def make_params(*, num_reqs, num_q_heads, num_kv_heads, head_dim, block_size, page_size, stride=None,
                total_tokens, max_seqlen, num_pages, max_pages_per_req, mask_pitch, budget_ppm=1_000_000,
                sm_scale=None, skip_delta=-1.0, flags=0) -> CosaParams:
    return CosaParams(
        num_reqs=num_reqs, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
        block_size=block_size, page_size=page_size, stride=stride if stride is not None else block_size // 8,
        total_tokens=total_tokens, max_seqlen=max_seqlen, num_pages=num_pages,
        max_pages_per_req=max_pages_per_req, mask_pitch=mask_pitch, budget_ppm=budget_ppm, flags=flags,
        sm_scale=float(sm_scale if sm_scale is not None else 1.0 / math.sqrt(head_dim)),
        skip_delta=float(skip_delta))


def stage1_pitch(budget_ppm: int, max_seqlen: int, block_size: int, top_p: bool = False) -> int:
    """Smallest mask pitch that holds K_i = ceil(B1 (i+1)) for every query block (with top-p, every
    causal candidate)."""
    nqb = -(-max_seqlen // block_size)
    return nqb if top_p else max(1, -(-budget_ppm * nqb // 1_000_000))


def cosa_proxy_workspace_size(p: CosaParams) -> int:
    return int(library().cosa_proxy_workspace_size(ctypes.byref(p)))


def cosa_prefill_workspace_size(p: CosaParams) -> int:
    return int(library().cosa_prefill_workspace_size(ctypes.byref(p)))


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def required_numel(p: CosaParams) -> dict:
    """Elements each buffer must hold at least, for the parameters ``p``, so that the library stays
    inside it (the layouts of include/cosa.h: q and out [T, Hq, d], caches [num_pages, P, Hkv, d],
    cu_seqlens [B + 1], page_table [B, max_pages_per_req], mask and visit_flags
    [B, Hq, nqb_max, mask_pitch], mask_len [B, Hq, nqb_max], status [1])."""
    nqb_max = -(-p.max_seqlen // p.block_size)
    rows = p.num_reqs * p.num_q_heads * nqb_max
    cache = p.num_pages * p.page_size * p.num_kv_heads * p.head_dim
    tokens = p.total_tokens * p.num_q_heads * p.head_dim
    return {"q": tokens, "out": tokens, "k_cache": cache, "v_cache": cache, "cu_seqlens": p.num_reqs + 1,
            "page_table": p.num_reqs * p.max_pages_per_req, "mask": rows * p.mask_pitch,
            "visit_flags": rows * p.mask_pitch, "mask_len": rows, "status": 1}


def validate_buffers(p: CosaParams, **buffers: Optional[torch.Tensor]) -> None:
    """Raise ValueError if a given buffer is smaller than the parameters say it is.  The library
    reads and writes the sizes ``p`` implies and cannot see the tensors' own sizes."""
    need = required_numel(p)
    for name, t in buffers.items():
        if t is not None and t.numel() < need[name]:
            raise ValueError(f"{name} holds {t.numel()} elements; the parameters need at least {need[name]}")


def params_for(q: torch.Tensor, k_cache: torch.Tensor, page_table: torch.Tensor, cu_seqlens: torch.Tensor, *,
               block_size: int, max_seqlen: int, stride: Optional[int] = None, budget_ppm: int = 1_000_000,
               mask_pitch: Optional[int] = None, skip_delta: float = -1.0,
               sm_scale: Optional[float] = None, flags: int = 0) -> CosaParams:
    T, Hq, d = q.shape
    num_pages, P, Hkv, d2 = k_cache.shape
    if d != d2:
        raise ValueError(f"q has head dim {d}, k_cache {d2}")
    B = cu_seqlens.numel() - 1
    if mask_pitch is None:
        mask_pitch = stage1_pitch(budget_ppm, max_seqlen, block_size)
    return make_params(num_reqs=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_size=block_size,
                       page_size=P, stride=stride, total_tokens=T, max_seqlen=max_seqlen, num_pages=num_pages,
                       max_pages_per_req=page_table.shape[1], mask_pitch=mask_pitch, budget_ppm=budget_ppm,
                       sm_scale=sm_scale, skip_delta=skip_delta, flags=flags)


def cosa_proxy_select(p: CosaParams, q: torch.Tensor, cu_seqlens: torch.Tensor, k_cache: torch.Tensor,
                      page_table: torch.Tensor, *, mask: Optional[torch.Tensor] = None,
                      mask_len: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      status: Optional[torch.Tensor] = None,
                      stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """KAP: returns (mask int32 [B, Hq, nqb_max, mask_pitch], mask_len int32 [B, Hq, nqb_max])."""
    _check(q, "q", torch.bfloat16)
    _check(k_cache, "k_cache", torch.bfloat16)
    _check(cu_seqlens, "cu_seqlens", torch.int32)
    _check(page_table, "page_table", torch.int32)
    for t, n in ((mask, "mask"), (mask_len, "mask_len"), (status, "status")):
        if t is not None:
            _check(t, n, torch.int32)
    validate_buffers(p, q=q, k_cache=k_cache, cu_seqlens=cu_seqlens, page_table=page_table, mask=mask,
                     mask_len=mask_len, status=status)
    dev = q.device
    nqb_max = -(-p.max_seqlen // p.block_size)
    if mask is None:
        mask = torch.empty((p.num_reqs, p.num_q_heads, nqb_max, p.mask_pitch), dtype=torch.int32, device=dev)
    if mask_len is None:
        mask_len = torch.empty((p.num_reqs, p.num_q_heads, nqb_max), dtype=torch.int32, device=dev)
    need = cosa_proxy_workspace_size(p)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    rc = library().cosa_proxy_select(ctypes.byref(p), _ptr(q), _ptr(cu_seqlens), _ptr(k_cache), _ptr(page_table),
                                     _ptr(mask), _ptr(mask_len), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(),
                                     _ptr(status), _stream_handle(stream))
    if rc != COSA_OK:
        raise CosaError(rc, "cosa_proxy_select")
    return mask, mask_len


def cosa_proxy_select_static(p: CosaParams, q: torch.Tensor, cu_seqlens: torch.Tensor, k_cache: torch.Tensor,
                             page_table: torch.Tensor, mask: torch.Tensor, mask_len: torch.Tensor, *,
                             status: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """KAP with the library's fixed device scratch instead of a workspace, for callers that cannot
    allocate device memory.  ``mask`` and ``mask_len`` are caller-owned outputs; nothing is allocated
    here.  Raises CosaError(COSA_ERR_WORKSPACE) when the problem needs more than STATIC_SCRATCH_BYTES."""
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (cu_seqlens, "cu_seqlens", torch.int32), (page_table, "page_table", torch.int32),
                     (mask, "mask", torch.int32), (mask_len, "mask_len", torch.int32)):
        _check(t, n, dt)
    if status is not None:
        _check(status, "status", torch.int32)
    validate_buffers(p, q=q, k_cache=k_cache, cu_seqlens=cu_seqlens, page_table=page_table, mask=mask,
                     mask_len=mask_len, status=status)
    rc = library().cosa_proxy_select_static(ctypes.byref(p), _ptr(q), _ptr(cu_seqlens), _ptr(k_cache),
                                            _ptr(page_table), _ptr(mask), _ptr(mask_len), _ptr(status),
                                            _stream_handle(stream))
    if rc != COSA_OK:
        raise CosaError(rc, "cosa_proxy_select_static")
    return mask, mask_len


def cosa_sparse_prefill(p: CosaParams, q: torch.Tensor, cu_seqlens: torch.Tensor, k_cache: torch.Tensor,
                        v_cache: torch.Tensor, page_table: torch.Tensor, mask: torch.Tensor,
                        mask_len: torch.Tensor, *, out: Optional[torch.Tensor] = None,
                        visit_flags: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                        status: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """OSK: returns out bf16 [T, Hq, d]; fills ``visit_flags`` (uint8, mask-shaped) if given."""
    for t, n, dt in ((q, "q", torch.bfloat16), (k_cache, "k_cache", torch.bfloat16),
                     (v_cache, "v_cache", torch.bfloat16), (cu_seqlens, "cu_seqlens", torch.int32),
                     (page_table, "page_table", torch.int32), (mask, "mask", torch.int32),
                     (mask_len, "mask_len", torch.int32)):
        _check(t, n, dt)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16)
    if visit_flags is not None:
        _check(visit_flags, "visit_flags", torch.uint8)
    if status is not None:
        _check(status, "status", torch.int32)
    validate_buffers(p, q=q, k_cache=k_cache, v_cache=v_cache, cu_seqlens=cu_seqlens, page_table=page_table,
                     mask=mask, mask_len=mask_len, out=out, visit_flags=visit_flags, status=status)
    need = cosa_prefill_workspace_size(p)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if need > ws_bytes:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        ws_bytes = need
    rc = library().cosa_sparse_prefill(ctypes.byref(p), _ptr(q), _ptr(cu_seqlens), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(page_table), _ptr(mask), _ptr(mask_len), _ptr(out), _ptr(visit_flags),
                                       _ptr(workspace), ws_bytes, _ptr(status), _stream_handle(stream))
    if rc != COSA_OK:
        raise CosaError(rc, "cosa_sparse_prefill")
    return out

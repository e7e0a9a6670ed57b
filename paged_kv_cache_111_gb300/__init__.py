"""Python binding of libpagedkv.so: paged KV-cache attention on one GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels behind the C ABI declared in ``include/pkv.h``; this module passes
torch tensors' device pointers, sizes and the current CUDA stream through
ctypes.  There is no fallback: if the library is missing or the tensors are
not on a CUDA device, the calls raise.

Calls (same names as the C ABI without the ``pkv_`` prefix):

* ``kv_write(kv_cache, key, value, slot_mapping, device_status=None)``
* ``paged_attn(out, query, kv_cache, block_tables, seq_lens, query_start_loc,
  max_query_len, max_seq_len, scale, workspace, num_splits=0)``
* ``paged_attn_combine(out, workspace)``
* ``copy_blocks(kv_cache, block_mapping)`` (copy-on-write of shared blocks)
* ``paged_attn_shared_prefix(..., shared_prefix_blocks, workspace)`` (cascade:
  a batch sharing a table prefix reads the shared blocks once)
* ``kv_write_fp8`` / ``paged_attn_fp8`` / ``paged_attn_shared_prefix_fp8`` (E4M3 cache with per-tensor
  K and V scales)

plus ``paged_attn_workspace_size(...)`` (the C call's size query) and
``workspace_status(workspace)`` (reads the device status word).
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import _build

__all__ = [
    "BLOCK_SIZE", "PagedKVError", "load", "kv_write", "paged_attn", "paged_attn_combine",
    "paged_attn_workspace_size", "workspace_status", "STATUS_NAMES", "library_path", "copy_blocks",
    "paged_attn_noalloc", "paged_attn_shared_prefix", "paged_attn_shared_prefix_workspace_size",
    "kv_write_fp8", "paged_attn_fp8", "paged_attn_shared_prefix_fp8", "workspace_schedule",
]

BLOCK_SIZE = 16
STATUS_NAMES = {
    0: "PKV_OK", 1: "PKV_ERR_NULL", 2: "PKV_ERR_SHAPE", 3: "PKV_ERR_UNSUPPORTED", 4: "PKV_ERR_ALIGNMENT",
    5: "PKV_ERR_WORKSPACE", 6: "PKV_ERR_CUDA", 7: "PKV_ERR_DEVICE_INDEX", 8: "PKV_ERR_DEVICE_METADATA",
    9: "PKV_ERR_DEVICE_TIMEOUT", 10: "PKV_ERR_PROTOCOL",
}

_lib = None
_lock = threading.Lock()


class PagedKVError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(code, code)}")
        self.code = code


def library_path() -> str:
    return _build.LIB


def load():
    """Load libpagedkv.so (built by ``__graft_entry__.build()`` or ``_build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise RuntimeError(
                f"{_build.LIB} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(_build.LIB)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.pkv_kv_write.argtypes = [P, i64, i32, i32, i32, P, i64, P, i64, P, i32, P, P]
        lib.pkv_kv_write.restype = ctypes.c_int
        lib.pkv_paged_attn.argtypes = [P, P, i64, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                       ctypes.c_float, i32, P, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t), P]
        lib.pkv_paged_attn.restype = ctypes.c_int
        lib.pkv_paged_attn_combine.argtypes = [P, P, ctypes.c_size_t, i32, i32, i32, P]
        lib.pkv_paged_attn_combine.restype = ctypes.c_int
        lib.pkv_copy_blocks.argtypes = [P, i64, i32, i32, i32, P, i32, P, P]
        lib.pkv_copy_blocks.restype = ctypes.c_int
        lib.pkv_paged_attn_shared_prefix.argtypes = [P, P, i64, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                                     i32, i32, ctypes.c_float, i32, i32, P, ctypes.c_size_t,
                                                     ctypes.POINTER(ctypes.c_size_t), P]
        lib.pkv_paged_attn_shared_prefix.restype = ctypes.c_int
        lib.pkv_kv_write_fp8.argtypes = [P, i64, i32, i32, i32, P, i64, P, i64, P, i32, ctypes.c_float,
                                         ctypes.c_float, P, P]
        lib.pkv_kv_write_fp8.restype = ctypes.c_int
        lib.pkv_paged_attn_fp8.argtypes = [P, P, i64, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32,
                                           i32, ctypes.c_float, ctypes.c_float, ctypes.c_float, i32, P,
                                           ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t), P]
        lib.pkv_paged_attn_fp8.restype = ctypes.c_int
        lib.pkv_paged_attn_shared_prefix_fp8.argtypes = [P, P, i64, P, i64, P, i32, P, P, i32, i32, i32, i32, i32,
                                                         i32, i32, i32, ctypes.c_float, ctypes.c_float,
                                                         ctypes.c_float, i32, i32, P, ctypes.c_size_t,
                                                         ctypes.POINTER(ctypes.c_size_t), P]
        lib.pkv_paged_attn_shared_prefix_fp8.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _need_cuda(*tensors: torch.Tensor) -> None:
    for t in tensors:
        if t is not None and not t.is_cuda:
            raise ValueError("paged KV-cache calls take CUDA tensors only")


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise PagedKVError(rc, what)


def kv_write(kv_cache: torch.Tensor, key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
             device_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Scatter key/value [T, Hkv, d] (bf16) into kv_cache [NB, Hkv, 2, 16, d] through slot_mapping [T] (int64)."""
    _need_cuda(kv_cache, key, value, slot_mapping, device_status)
    nb, hkv, _, bs, d = kv_cache.shape
    T = int(slot_mapping.shape[0])
    if key.dim() != 3 or key.stride(2) != 1 or key.stride(1) != d or value.stride(2) != 1 or value.stride(1) != d:
        raise ValueError("key/value must be [T, Hkv, d] with contiguous heads")
    rc = load().pkv_kv_write(_ptr(kv_cache), nb, hkv, d, bs, _ptr(key), key.stride(0), _ptr(value),
                             value.stride(0), _ptr(slot_mapping), T, _ptr(device_status), _stream(kv_cache, stream))
    _check(rc, "pkv_kv_write")


def copy_blocks(kv_cache: torch.Tensor, block_mapping: torch.Tensor, device_status: Optional[torch.Tensor] = None,
                stream=None) -> None:
    """Copy-on-write: block_mapping int64 [num_pairs, 2] of {source, destination} block ids."""
    _need_cuda(kv_cache, block_mapping, device_status)
    nb, hkv, _, bs, d = kv_cache.shape
    if block_mapping.dim() != 2 or block_mapping.shape[1] != 2 or not block_mapping.is_contiguous():
        raise ValueError("block_mapping must be a contiguous [num_pairs, 2] int64 tensor")
    rc = load().pkv_copy_blocks(_ptr(kv_cache), nb, hkv, d, bs, _ptr(block_mapping), int(block_mapping.shape[0]),
                                _ptr(device_status), _stream(kv_cache, stream))
    _check(rc, "pkv_copy_blocks")


def paged_attn_workspace_size(num_seqs: int, num_tokens: int, max_query_len: int, max_seq_len: int,
                              num_q_heads: int, num_kv_heads: int, head_size: int) -> int:
    """Bytes of workspace pkv_paged_attn needs for these sizes (no GPU work)."""
    need = ctypes.c_size_t(0)
    max_blocks = (max_seq_len + BLOCK_SIZE - 1) // BLOCK_SIZE
    rc = load().pkv_paged_attn(None, None, num_q_heads * head_size, None, 1, None, max_blocks, None, None,
                               num_seqs, num_tokens, max_query_len, max_seq_len, num_q_heads, num_kv_heads,
                               head_size, BLOCK_SIZE, ctypes.c_float(1.0), 0, None, 0, ctypes.byref(need), None)
    if rc not in (0, 1, 5):
        _check(rc, "pkv_paged_attn (size query)")
    return int(need.value)


def paged_attn(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor, block_tables: torch.Tensor,
               seq_lens: torch.Tensor, query_start_loc: torch.Tensor, max_query_len: int, max_seq_len: int,
               scale: float, workspace: torch.Tensor, num_splits: int = 0, stream=None) -> None:
    """Causal paged attention; out [T, H, d] bf16.  Follow with paged_attn_combine on the same stream."""
    _need_cuda(out, query, kv_cache, block_tables, seq_lens, query_start_loc, workspace)
    nb, hkv, _, bs, d = kv_cache.shape
    T, H = int(query.shape[0]), int(query.shape[1])
    if query.stride(2) != 1 or query.stride(1) != d:
        raise ValueError("query must be [T, H, d] with contiguous heads")
    if not out.is_contiguous() or tuple(out.shape) != (T, H, d):
        raise ValueError("out must be a contiguous [T, H, d] tensor")
    if block_tables.dim() != 2 or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous [num_seqs, max_blocks] tensor")
    S = int(seq_lens.shape[0])
    need = ctypes.c_size_t(0)
    rc = load().pkv_paged_attn(_ptr(out), _ptr(query), query.stride(0), _ptr(kv_cache), nb, _ptr(block_tables),
                               int(block_tables.shape[1]), _ptr(seq_lens), _ptr(query_start_loc), S, T,
                               int(max_query_len), int(max_seq_len), H, hkv, d, bs, ctypes.c_float(scale),
                               int(num_splits), _ptr(workspace), workspace.numel() * workspace.element_size(),
                               ctypes.byref(need), _stream(out, stream))
    _check(rc, "pkv_paged_attn")


def paged_attn_shared_prefix_workspace_size(num_seqs: int, num_tokens: int, max_query_len: int, max_seq_len: int,
                                            num_q_heads: int, num_kv_heads: int, head_size: int,
                                            shared_prefix_blocks: int) -> int:
    """Bytes of workspace pkv_paged_attn_shared_prefix needs (no GPU work)."""
    need = ctypes.c_size_t(0)
    max_blocks = max((max_seq_len + BLOCK_SIZE - 1) // BLOCK_SIZE, shared_prefix_blocks)
    rc = load().pkv_paged_attn_shared_prefix(None, None, num_q_heads * head_size, None, 1, None, max_blocks, None,
                                             None, num_seqs, num_tokens, max_query_len, max_seq_len, num_q_heads,
                                             num_kv_heads, head_size, BLOCK_SIZE, ctypes.c_float(1.0), 0,
                                             shared_prefix_blocks, None, 0, ctypes.byref(need), None)
    if rc not in (0, 1, 5):
        _check(rc, "pkv_paged_attn_shared_prefix (size query)")
    return int(need.value)


def paged_attn_shared_prefix(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor,
                             block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                             max_query_len: int, max_seq_len: int, scale: float, shared_prefix_blocks: int,
                             workspace: torch.Tensor, num_splits: int = 0, stream=None) -> None:
    """paged_attn with the first shared_prefix_blocks table entries shared by the batch (cascade)."""
    _need_cuda(out, query, kv_cache, block_tables, seq_lens, query_start_loc, workspace)
    nb, hkv, _, bs, d = kv_cache.shape
    T, H = int(query.shape[0]), int(query.shape[1])
    if query.stride(2) != 1 or query.stride(1) != d:
        raise ValueError("query must be [T, H, d] with contiguous heads")
    if not out.is_contiguous() or tuple(out.shape) != (T, H, d):
        raise ValueError("out must be a contiguous [T, H, d] tensor")
    if block_tables.dim() != 2 or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous [num_seqs, max_blocks] tensor")
    need = ctypes.c_size_t(0)
    rc = load().pkv_paged_attn_shared_prefix(
        _ptr(out), _ptr(query), query.stride(0), _ptr(kv_cache), nb, _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(seq_lens), _ptr(query_start_loc), int(seq_lens.shape[0]), T, int(max_query_len), int(max_seq_len), H,
        hkv, d, bs, ctypes.c_float(scale), int(num_splits), int(shared_prefix_blocks), _ptr(workspace),
        workspace.numel() * workspace.element_size(), ctypes.byref(need), _stream(out, stream))
    _check(rc, "pkv_paged_attn_shared_prefix")


def kv_write_fp8(kv_cache: torch.Tensor, key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
                 k_scale: float, v_scale: float, device_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """kv_write into an E4M3 cache (uint8 or float8_e4m3fn [NB, Hkv, 2, 16, d]): code = E4M3(x / scale)."""
    _need_cuda(kv_cache, key, value, slot_mapping, device_status)
    if kv_cache.element_size() != 1:
        raise ValueError("an FP8 cache holds one byte per element")
    nb, hkv, _, bs, d = kv_cache.shape
    T = int(slot_mapping.shape[0])
    if key.dim() != 3 or key.stride(2) != 1 or key.stride(1) != d or value.stride(2) != 1 or value.stride(1) != d:
        raise ValueError("key/value must be [T, Hkv, d] with contiguous heads")
    rc = load().pkv_kv_write_fp8(_ptr(kv_cache), nb, hkv, d, bs, _ptr(key), key.stride(0), _ptr(value),
                                 value.stride(0), _ptr(slot_mapping), T, ctypes.c_float(k_scale),
                                 ctypes.c_float(v_scale), _ptr(device_status), _stream(kv_cache, stream))
    _check(rc, "pkv_kv_write_fp8")


def paged_attn_fp8(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor, block_tables: torch.Tensor,
                   seq_lens: torch.Tensor, query_start_loc: torch.Tensor, max_query_len: int, max_seq_len: int,
                   scale: float, k_scale: float, v_scale: float, workspace: torch.Tensor, num_splits: int = 0,
                   stream=None) -> None:
    """paged_attn over an E4M3 cache; the workspace is sized as for paged_attn."""
    _need_cuda(out, query, kv_cache, block_tables, seq_lens, query_start_loc, workspace)
    if kv_cache.element_size() != 1:
        raise ValueError("an FP8 cache holds one byte per element")
    nb, hkv, _, bs, d = kv_cache.shape
    T, H = int(query.shape[0]), int(query.shape[1])
    if query.stride(2) != 1 or query.stride(1) != d:
        raise ValueError("query must be [T, H, d] with contiguous heads")
    if not out.is_contiguous() or tuple(out.shape) != (T, H, d):
        raise ValueError("out must be a contiguous [T, H, d] tensor")
    if block_tables.dim() != 2 or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous [num_seqs, max_blocks] tensor")
    need = ctypes.c_size_t(0)
    rc = load().pkv_paged_attn_fp8(
        _ptr(out), _ptr(query), query.stride(0), _ptr(kv_cache), nb, _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(seq_lens), _ptr(query_start_loc), int(seq_lens.shape[0]), T, int(max_query_len), int(max_seq_len), H,
        hkv, d, bs, ctypes.c_float(scale), ctypes.c_float(k_scale), ctypes.c_float(v_scale), int(num_splits),
        _ptr(workspace), workspace.numel() * workspace.element_size(), ctypes.byref(need), _stream(out, stream))
    _check(rc, "pkv_paged_attn_fp8")


def paged_attn_shared_prefix_fp8(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor,
                                 block_tables: torch.Tensor, seq_lens: torch.Tensor, query_start_loc: torch.Tensor,
                                 max_query_len: int, max_seq_len: int, scale: float, k_scale: float, v_scale: float,
                                 shared_prefix_blocks: int, workspace: torch.Tensor, num_splits: int = 0,
                                 stream=None) -> None:
    """paged_attn_shared_prefix over an E4M3 cache; the workspace is sized as for paged_attn_shared_prefix."""
    _need_cuda(out, query, kv_cache, block_tables, seq_lens, query_start_loc, workspace)
    if kv_cache.element_size() != 1:
        raise ValueError("an FP8 cache holds one byte per element")
    nb, hkv, _, bs, d = kv_cache.shape
    T, H = int(query.shape[0]), int(query.shape[1])
    if query.stride(2) != 1 or query.stride(1) != d:
        raise ValueError("query must be [T, H, d] with contiguous heads")
    if not out.is_contiguous() or tuple(out.shape) != (T, H, d):
        raise ValueError("out must be a contiguous [T, H, d] tensor")
    if block_tables.dim() != 2 or not block_tables.is_contiguous():
        raise ValueError("block_tables must be a contiguous [num_seqs, max_blocks] tensor")
    need = ctypes.c_size_t(0)
    rc = load().pkv_paged_attn_shared_prefix_fp8(
        _ptr(out), _ptr(query), query.stride(0), _ptr(kv_cache), nb, _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(seq_lens), _ptr(query_start_loc), int(seq_lens.shape[0]), T, int(max_query_len), int(max_seq_len), H,
        hkv, d, bs, ctypes.c_float(scale), ctypes.c_float(k_scale), ctypes.c_float(v_scale), int(num_splits),
        int(shared_prefix_blocks), _ptr(workspace), workspace.numel() * workspace.element_size(),
        ctypes.byref(need), _stream(out, stream))
    _check(rc, "pkv_paged_attn_shared_prefix_fp8")


def paged_attn_combine(out: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Log-sum-exp merge of the rows pkv_paged_attn split; out as given to paged_attn."""
    _need_cuda(out, workspace)
    T, H, d = out.shape
    rc = load().pkv_paged_attn_combine(_ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       T, H, d, _stream(out, stream))
    _check(rc, "pkv_paged_attn_combine")


def workspace_status(workspace: torch.Tensor) -> int:
    """The device status word (first int32 of the workspace); synchronises on its read."""
    return int(workspace[:4].view(torch.int32)[0].item())


# per-CTA record of the persistent prefill kernels' dynamic schedule: int32
# [2][1024] right after the workspace's 256-byte header
_SCHEDULE_OFFSET, _SCHEDULE_CTAS = 256, 1024


def workspace_schedule(workspace: torch.Tensor):
    """Work items each CTA of the tensor-core prefill kernel (first list) and of
    the shared-prefix pass (second list) took in the last attention call on
    this workspace, trailing idle CTAs dropped; synchronises on its read."""
    a = workspace[_SCHEDULE_OFFSET:_SCHEDULE_OFFSET + 8 * _SCHEDULE_CTAS].view(torch.int32).cpu().tolist()

    def trim(v):
        while v and v[-1] == 0:
            v.pop()
        return v
    return trim(a[:_SCHEDULE_CTAS]), trim(a[_SCHEDULE_CTAS:])


def paged_attn_noalloc(out: torch.Tensor, query: torch.Tensor, kv_cache: torch.Tensor, block_tables: torch.Tensor,
                       seq_lens: torch.Tensor, query_start_loc: torch.Tensor, max_query_len: int, max_seq_len: int,
                       scale: float, num_splits: int = 0, device_status: Optional[torch.Tensor] = None,
                       stream=None) -> None:
    """paged_attn + paged_attn_combine without a caller workspace: for callers
    that cannot allocate device memory.  The scratch is the library's own
    fixed device array (see pkv_paged_attn_noalloc in include/pkv.h)."""
    _need_cuda(out, query, kv_cache, block_tables, seq_lens, query_start_loc, device_status)
    lib = load()
    fn = lib.pkv_paged_attn_noalloc
    if fn.argtypes is None:
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        fn.argtypes = [P, P, i64, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i32,
                       ctypes.c_float, i32, P, P]
        fn.restype = ctypes.c_int
    nb, hkv, _, bs, d = kv_cache.shape
    T, H = int(query.shape[0]), int(query.shape[1])
    if query.stride(2) != 1 or query.stride(1) != d:
        raise ValueError("query must be [T, H, d] with contiguous heads")
    if not out.is_contiguous() or tuple(out.shape) != (T, H, d):
        raise ValueError("out must be a contiguous [T, H, d] tensor")
    rc = fn(_ptr(out), _ptr(query), query.stride(0), _ptr(kv_cache), nb, _ptr(block_tables),
            int(block_tables.shape[1]), _ptr(seq_lens), _ptr(query_start_loc), int(seq_lens.shape[0]), T,
            int(max_query_len), int(max_seq_len), H, hkv, d, bs, ctypes.c_float(scale), int(num_splits),
            _ptr(device_status), _stream(out, stream))
    _check(rc, "pkv_paged_attn_noalloc")

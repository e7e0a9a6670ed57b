"""CPU oracle for paged KV-cache attention (fp64, plain C).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The product library never loads
this module, and this module never loads the product library.

``build()`` compiles ``pkv_oracle.c`` with gcc (OpenMP when available) into
``liboracle.so`` beside it.  The wrappers below take CPU torch tensors or
numpy arrays and marshal them to the C functions; every bit of arithmetic
lives in the C file.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {-1: "invalid argument", -2: "index out of range", -3: "duplicate slot", -4: "out of memory"}


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle if it is missing or older than its source."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O3", "-std=c11", "-shared", "-fPIC", "-Wall", "-o", tmp, _SRC]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:] + ["-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_kv_write.argtypes = [P, i64, i32, i32, i32, P, P, P, i32]
            lib.oracle_kv_write.restype = ctypes.c_int
            lib.oracle_paged_attn.argtypes = [P, P, P, P, i64, P, i32, P, P, i32,
                                              i32, i32, i32, i32, f32, i32]
            lib.oracle_paged_attn.restype = ctypes.c_int
            lib.oracle_attn_row.argtypes = [P, P, P, P, P, i64, P, i32, P, P, i32,
                                            i32, i32, i32, i32, f32, i32, i32, i32, i64, i64]
            lib.oracle_attn_row.restype = ctypes.c_int
            lib.oracle_lse_combine.argtypes = [P, P, P, P, i32, i32]
            lib.oracle_lse_combine.restype = ctypes.c_int
            lib.oracle_copy_blocks.argtypes = [P, i64, i32, i32, i32, P, i32]
            lib.oracle_copy_blocks.restype = ctypes.c_int
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_encode.argtypes = [f32]
            lib.oracle_e4m3_encode.restype = ctypes.c_uint8
            lib.oracle_kv_write_fp8.argtypes = [P, i64, i32, i32, i32, P, P, P, i32, f32, f32]
            lib.oracle_kv_write_fp8.restype = ctypes.c_int
            lib.oracle_paged_attn_fp8.argtypes = [P, P, P, P, i64, P, i32, P, P, i32,
                                                  i32, i32, i32, i32, f32, f32, f32, i32]
            lib.oracle_paged_attn_fp8.restype = ctypes.c_int
            _lib = lib
    return _lib


class use_library:
    """Temporarily route every wrapper to another build of the oracle source.

    Used by the tests that plant a mistake in a copy of the oracle and check
    that the pins catch it.
    """

    def __init__(self, path: str):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        self.saved = _load()
        lib = ctypes.CDLL(self.path)
        for name in ("oracle_max_threads", "oracle_kv_write", "oracle_paged_attn",
                     "oracle_attn_row", "oracle_lse_combine", "oracle_copy_blocks",
                     "oracle_e4m3_decode", "oracle_e4m3_encode", "oracle_kv_write_fp8",
                     "oracle_paged_attn_fp8"):
            src, dst = getattr(self.saved, name), getattr(lib, name)
            dst.restype = src.restype
            if src.argtypes is not None:
                dst.argtypes = src.argtypes
        with _lock:
            _lib = lib
        return lib

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self.saved
        return False


def _np(x, dtype) -> np.ndarray:
    """A C-contiguous numpy view/copy of a CPU torch tensor or array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            if x.dtype == torch.bfloat16:
                x = x.contiguous().view(torch.int16).numpy().view(np.uint16)
            else:
                x = x.contiguous().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a.size else None


def _check(rc: int, what: str) -> int:
    if rc < 0:
        raise OracleError(f"{what}: {ERRORS.get(rc, rc)}")
    return rc


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def new_cache(num_blocks: int, num_kv_heads: int, head_size: int, block_size: int = 16) -> np.ndarray:
    """A cache of raw bf16 bit patterns, all bf16 NaN (0x7FC0)."""
    return np.full((num_blocks, num_kv_heads, 2, block_size, head_size), 0x7FC0, dtype=np.uint16)


def kv_write(cache: np.ndarray, key, value, slot_mapping) -> None:
    """In-place cache write (bit copy) of key/value [T, Hkv, d] through slot_mapping [T]."""
    nb, hkv, two, bs, d = cache.shape
    assert cache.dtype == np.uint16 and cache.flags.c_contiguous and two == 2
    k = _np(key, np.uint16)
    v = _np(value, np.uint16)
    s = _np(slot_mapping, np.int64)
    T = int(s.shape[0])
    assert k.shape == (T, hkv, d) and v.shape == (T, hkv, d)
    _check(_load().oracle_kv_write(_ptr(cache), nb, hkv, d, bs, _ptr(k), _ptr(v), _ptr(s), T),
           "oracle_kv_write")


def copy_blocks(cache: np.ndarray, mapping) -> None:
    """In-place copy-on-write block copies; mapping int64 [n, 2] of {source, destination}."""
    nb, hkv, _, bs, d = cache.shape
    m = _np(mapping, np.int64).reshape(-1, 2)
    _check(_load().oracle_copy_blocks(_ptr(cache), nb, hkv, d, bs, _ptr(m), int(m.shape[0])),
           "oracle_copy_blocks")


def paged_attn(cache: np.ndarray, query, block_tables, seq_lens, query_start_loc,
               num_q_heads: int, scale: float, num_threads: int = 0):
    """Attention of every query row; returns (out [T, H, d] fp64, lse [T, H] fp64)."""
    nb, hkv, _, bs, d = cache.shape
    q = _np(query, np.uint16)
    bt = _np(block_tables, np.int32)
    sl = _np(seq_lens, np.int32)
    qsl = _np(query_start_loc, np.int32)
    S = int(sl.shape[0])
    T = int(qsl[-1]) if S else 0
    out = np.zeros((T, num_q_heads, d), dtype=np.float64)
    lse = np.zeros((T, num_q_heads), dtype=np.float64)
    maxb = int(bt.shape[1]) if bt.ndim == 2 else 0
    _check(_load().oracle_paged_attn(_ptr(out), _ptr(lse), _ptr(q), _ptr(cache), nb, _ptr(bt), maxb,
                                     _ptr(sl), _ptr(qsl), S, num_q_heads, hkv, d, bs,
                                     ctypes.c_float(scale), int(num_threads)),
           "oracle_paged_attn")
    return out, lse


def attn_row(cache: np.ndarray, query, block_tables, seq_lens, query_start_loc,
             num_q_heads: int, scale: float, request: int, query_index: int, q_head: int,
             key_begin: int = 0, key_end: Optional[int] = None, want_weights: bool = False):
    """One row over keys [key_begin, key_end): returns (out [d], lse, weights or None)."""
    nb, hkv, _, bs, d = cache.shape
    q = _np(query, np.uint16)
    bt = _np(block_tables, np.int32)
    sl = _np(seq_lens, np.int32)
    qsl = _np(query_start_loc, np.int32)
    if key_end is None:
        key_end = int(sl[request])
    out = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    w = np.zeros(max(1, key_end - key_begin), dtype=np.float64) if want_weights else None
    n = _check(_load().oracle_attn_row(_ptr(out), _ptr(lse), _ptr(w) if w is not None else None,
                                       _ptr(q), _ptr(cache), nb, _ptr(bt), int(bt.shape[1]),
                                       _ptr(sl), _ptr(qsl), int(sl.shape[0]), num_q_heads, hkv, d, bs,
                                       ctypes.c_float(scale), request, query_index, q_head,
                                       key_begin, key_end),
               "oracle_attn_row")
    return out, float(lse[0]), (w[:n] if w is not None else None)


def lse_combine(part_out, part_lse):
    """Merge partial (out [n, d], lse [n]) over a partition of keys; returns (out [d], lse)."""
    po = np.ascontiguousarray(part_out, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    n, d = po.shape
    out = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _check(_load().oracle_lse_combine(_ptr(out), _ptr(lse), _ptr(po), _ptr(pl), n, d),
           "oracle_lse_combine")
    return out, float(lse[0])


def run_step(step, num_threads: int = 0):
    """Build the oracle's own cache for a ``workloads.Step`` and run the step.

    The cache starts all-NaN; the history entries and then the step's new
    tokens are written with the oracle's kv_write, and attention follows.
    Returns (cache, out fp64 [T, H, d], lse fp64 [T, H]).
    """
    cache = new_cache(step.num_blocks, step.num_kv_heads, step.head_size, step.block_size)
    kv_write(cache, step.hist_key, step.hist_value, step.hist_slot_mapping)
    kv_write(cache, step.key, step.value, step.slot_mapping)
    out, lse = paged_attn(cache, step.query, step.block_tables, step.seq_lens,
                          step.query_start_loc, step.num_q_heads, step.scale, num_threads)
    return cache, out, lse


# ---- FP8 (E4M3) cache ---------------------------------------------------------

E4M3_NAN = 0x7F


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (NaN for 0x7F / 0xFF)."""
    return float(_load().oracle_e4m3_decode(int(code) & 0xFF))


def e4m3_encode(x: float) -> int:
    """Nearest E4M3 code of the fp32 value x (ties to even, held at +-448)."""
    return int(_load().oracle_e4m3_encode(ctypes.c_float(x)))


def new_cache_fp8(num_blocks: int, num_kv_heads: int, head_size: int, block_size: int = 16) -> np.ndarray:
    """An E4M3 cache of raw bytes, all NaN (0x7F)."""
    return np.full((num_blocks, num_kv_heads, 2, block_size, head_size), E4M3_NAN, dtype=np.uint8)


def kv_write_fp8(cache: np.ndarray, key, value, slot_mapping, k_scale: float, v_scale: float) -> None:
    """In-place write of bf16 key/value [T, Hkv, d] into an E4M3 cache: code = E4M3(x / scale)."""
    nb, hkv, two, bs, d = cache.shape
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous and two == 2
    k = _np(key, np.uint16)
    v = _np(value, np.uint16)
    s = _np(slot_mapping, np.int64)
    T = int(s.shape[0])
    assert k.shape == (T, hkv, d) and v.shape == (T, hkv, d)
    _check(_load().oracle_kv_write_fp8(_ptr(cache), nb, hkv, d, bs, _ptr(k), _ptr(v), _ptr(s), T,
                                       ctypes.c_float(k_scale), ctypes.c_float(v_scale)),
           "oracle_kv_write_fp8")


def paged_attn_fp8(cache: np.ndarray, query, block_tables, seq_lens, query_start_loc,
                   num_q_heads: int, scale: float, k_scale: float, v_scale: float, num_threads: int = 0):
    """Attention over an E4M3 cache (values code * scale); returns (out fp64, lse fp64)."""
    nb, hkv, _, bs, d = cache.shape
    assert cache.dtype == np.uint8
    q = _np(query, np.uint16)
    bt = _np(block_tables, np.int32)
    sl = _np(seq_lens, np.int32)
    qsl = _np(query_start_loc, np.int32)
    S = int(sl.shape[0])
    T = int(qsl[-1]) if S else 0
    out = np.zeros((T, num_q_heads, d), dtype=np.float64)
    lse = np.zeros((T, num_q_heads), dtype=np.float64)
    maxb = int(bt.shape[1]) if bt.ndim == 2 else 0
    _check(_load().oracle_paged_attn_fp8(_ptr(out), _ptr(lse), _ptr(q), _ptr(cache), nb, _ptr(bt), maxb,
                                         _ptr(sl), _ptr(qsl), S, num_q_heads, hkv, d, bs,
                                         ctypes.c_float(scale), ctypes.c_float(k_scale),
                                         ctypes.c_float(v_scale), int(num_threads)),
           "oracle_paged_attn_fp8")
    return out, lse


def run_step_fp8(step, k_scale: float, v_scale: float, num_threads: int = 0):
    """run_step over an E4M3 cache: (cache uint8, out fp64 [T, H, d], lse fp64 [T, H])."""
    cache = new_cache_fp8(step.num_blocks, step.num_kv_heads, step.head_size, step.block_size)
    kv_write_fp8(cache, step.hist_key, step.hist_value, step.hist_slot_mapping, k_scale, v_scale)
    kv_write_fp8(cache, step.key, step.value, step.slot_mapping, k_scale, v_scale)
    out, lse = paged_attn_fp8(cache, step.query, step.block_tables, step.seq_lens,
                              step.query_start_loc, step.num_q_heads, step.scale, k_scale, v_scale,
                              num_threads)
    return cache, out, lse

"""The C ABI without a GPU: the library builds, loads and exports every
declared entry point, and host-side argument checks return their codes
before anything is enqueued (no CUDA call is reached)."""

import ctypes
import glob
import os
import re
import subprocess

import pytest

import paged_kv_cache_111_gb300 as pkv
from paged_kv_cache_111_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return pkv.load()


def declared_symbols():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        with open(h) as f:
            text = f.read()
        names |= set(re.findall(r"^\s*int\s+(pkv_\w+)\s*\(", text, flags=re.M))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"pkv_kv_write", "pkv_paged_attn", "pkv_paged_attn_combine"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT\s+(pkv_\w+)", out.stdout))
    for n in names:
        assert n in exported, f"{n} declared in include/ but not exported"
        assert getattr(lib, n) is not None


def test_oracle_and_library_share_nothing():
    """The oracle never includes the library's headers or sources, and the
    library never includes anything under oracle/."""
    with open(os.path.join(ROOT, "oracle", "pkv_oracle.c")) as f:
        osrc = f.read()
    assert "pkv.h" not in osrc and "pkv_common" not in osrc
    for src in glob.glob(os.path.join(ROOT, "paged_kv_cache_111_gb300", "**", "*"), recursive=True):
        if src.endswith((".cu", ".cuh", ".py", ".h", ".cpp")):
            with open(src) as f:
                text = f.read()
            assert "oracle" not in re.sub(r"(?m)^\s*(//|#).*$", "", text).lower(), src


def test_kv_write_argument_errors(lib):
    P = ctypes.c_void_p
    fake = P(0x10000)          # never dereferenced: validation fails first
    s = ctypes.c_void_p(0x20000)
    assert lib.pkv_kv_write(fake, 4, 2, 96, 16, fake, 256, fake, 256, s, 3, None, None) == 3
    assert lib.pkv_kv_write(fake, 4, 2, 128, 32, fake, 256, fake, 256, s, 3, None, None) == 3
    assert lib.pkv_kv_write(fake, 4, 0, 128, 16, fake, 256, fake, 256, s, 3, None, None) == 2
    assert lib.pkv_kv_write(None, 4, 2, 128, 16, fake, 256, fake, 256, s, 3, None, None) == 1
    assert lib.pkv_kv_write(P(0x10002), 4, 2, 128, 16, fake, 256, fake, 256, s, 3, None, None) == 4
    assert lib.pkv_kv_write(fake, 4, 2, 128, 16, fake, 100, fake, 256, s, 3, None, None) == 2
    assert lib.pkv_kv_write(fake, 4, 2, 128, 16, fake, 260, fake, 256, s, 3, None, None) == 4
    assert lib.pkv_kv_write(fake, 4, 2, 128, 16, fake, 256, fake, 256, s, 0, None, None) == 0


def _attn(lib, **kw):
    a = dict(out=0x10000, query=0x10000, qstride=512, cache=0x10000, nb=16, bt=0x20000, maxb=4, sl=0x20000,
             qsl=0x20000, S=2, T=2, maxq=1, maxs=64, H=4, Hkv=2, d=128, bs=16, scale=0.125, splits=0,
             ws=None, wsb=0)
    a.update(kw)
    need = ctypes.c_size_t(0)
    P = ctypes.c_void_p
    rc = lib.pkv_paged_attn(P(a["out"]) if a["out"] else None, P(a["query"]) if a["query"] else None,
                            a["qstride"], P(a["cache"]) if a["cache"] else None, a["nb"], P(a["bt"]),
                            a["maxb"], P(a["sl"]), P(a["qsl"]), a["S"], a["T"], a["maxq"], a["maxs"], a["H"],
                            a["Hkv"], a["d"], a["bs"], ctypes.c_float(a["scale"]), a["splits"],
                            P(a["ws"]) if a["ws"] else None, a["wsb"], ctypes.byref(need), None)
    return rc, need.value


def test_paged_attn_argument_errors_and_size_query(lib):
    rc, need = _attn(lib)
    assert rc == 5 and need > 256                       # the size query
    assert _attn(lib, d=96)[0] == 3
    assert _attn(lib, bs=32)[0] == 3
    assert _attn(lib, H=3)[0] == 2                      # q heads not a multiple of kv heads
    assert _attn(lib, maxb=3)[0] == 2                   # table too short for max_seq_len
    assert _attn(lib, S=0, T=2)[0] == 2                 # tokens without requests
    assert _attn(lib, maxq=65)[0] == 2
    assert _attn(lib, out=None)[0] == 1
    assert _attn(lib, scale=float("nan"))[0] == 2
    assert _attn(lib, nb=1 << 30, Hkv=2, H=4)[0] == 2   # blocks x kv heads past 2^31 - 1
    assert _attn(lib, ws=0x40000, wsb=need - 1)[0] == 5
    assert _attn(lib, ws=0x40010, wsb=need)[0] == 4     # workspace not 256-byte aligned
    assert _attn(lib, qstride=500, ws=0x40000, wsb=need)[0] == 2
    assert _attn(lib, qstride=516, ws=0x40000, wsb=need)[0] == 4
    assert _attn(lib, S=0, T=0)[0] == 0                 # nothing to do


def test_workspace_grows_with_the_hints(lib):
    a = _attn(lib, maxs=64)[1]
    b = _attn(lib, maxs=4096, maxb=256)[1]
    c = _attn(lib, S=256, T=256, maxs=4096, maxb=256)[1]
    assert a < b < c
    # a decode batch at the 13B shape needs under 1% of the 32.8 GB cache it reads
    n = pkv.paged_attn_workspace_size(256, 256, 1, 4096, 40, 40, 128)
    assert n < 100000 * 40 * 2 * 16 * 128 * 2 // 100


def test_combine_argument_errors(lib):
    P = ctypes.c_void_p
    assert lib.pkv_paged_attn_combine(P(0x10000), P(0x40000), 1 << 20, 2, 4, 96, None) == 3
    assert lib.pkv_paged_attn_combine(None, P(0x40000), 1 << 20, 2, 4, 128, None) == 1
    assert lib.pkv_paged_attn_combine(P(0x10000), P(0x40000), 100, 2, 4, 128, None) == 5
    assert lib.pkv_paged_attn_combine(P(0x10000), P(0x40010), 1 << 20, 2, 4, 128, None) == 4
    assert lib.pkv_paged_attn_combine(P(0x10000), P(0x40000), 1 << 20, 0, 4, 128, None) == 0


def test_binding_refuses_cpu_tensors():
    import torch
    t = torch.zeros(1, 2, 2, 16, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        pkv.kv_write(t, torch.zeros(1, 2, 64, dtype=torch.bfloat16), torch.zeros(1, 2, 64, dtype=torch.bfloat16),
                     torch.zeros(1, dtype=torch.int64))


def _attn_variant(fn, lib, extra_before_splits=(), extra_after_splits=(), **kw):
    """pkv_paged_attn's argument list for the E4M3 / shared-prefix variants:
    `extra_before_splits` go after the scale (k_scale, v_scale), the others
    after num_splits (shared_prefix_blocks)."""
    a = dict(out=0x10000, query=0x10000, qstride=512, cache=0x10000, nb=16, bt=0x20000, maxb=4, sl=0x20000,
             qsl=0x20000, S=2, T=2, maxq=1, maxs=64, H=4, Hkv=2, d=128, bs=16, scale=0.125, splits=0,
             ws=None, wsb=0)
    a.update(kw)
    need = ctypes.c_size_t(0)
    P = ctypes.c_void_p
    rc = getattr(lib, fn)(P(a["out"]), P(a["query"]), a["qstride"], P(a["cache"]), a["nb"], P(a["bt"]), a["maxb"],
                          P(a["sl"]), P(a["qsl"]), a["S"], a["T"], a["maxq"], a["maxs"], a["H"], a["Hkv"], a["d"],
                          a["bs"], ctypes.c_float(a["scale"]), *extra_before_splits, a["splits"],
                          *extra_after_splits, P(a["ws"]) if a["ws"] else None, a["wsb"], ctypes.byref(need), None)
    return rc, need.value


def test_fp8_argument_errors(lib):
    P = ctypes.c_void_p
    fake, s = P(0x10000), P(0x20000)
    f = ctypes.c_float
    # the cache write: scales must be positive and finite
    for ks, vs in ((0.0, 1.0), (1.0, -1.0), (float("nan"), 1.0), (1.0, float("inf"))):
        assert lib.pkv_kv_write_fp8(fake, 4, 2, 128, 16, fake, 256, fake, 256, s, 3, f(ks), f(vs), None, None) == 2
    assert lib.pkv_kv_write_fp8(fake, 4, 2, 96, 16, fake, 256, fake, 256, s, 3, f(1), f(1), None, None) == 3
    assert lib.pkv_kv_write_fp8(None, 4, 2, 128, 16, fake, 256, fake, 256, s, 3, f(1), f(1), None, None) == 1
    assert lib.pkv_kv_write_fp8(fake, 4, 2, 128, 16, fake, 256, fake, 256, s, 0, f(1), f(1), None, None) == 0
    # attention: the same scale rule, the same size query as the bf16 call
    good = (f(0.02), f(0.03))
    rc, need = _attn_variant("pkv_paged_attn_fp8", lib, good)
    assert rc == 5 and need == _attn(lib)[1]
    for ks, vs in ((0.0, 1.0), (1.0, float("nan")), (float("inf"), 1.0)):
        assert _attn_variant("pkv_paged_attn_fp8", lib, (f(ks), f(vs)))[0] == 2
    assert _attn_variant("pkv_paged_attn_fp8", lib, good, d=96)[0] == 3
    assert _attn_variant("pkv_paged_attn_fp8", lib, good, out=0)[0] == 1


def test_shared_prefix_argument_errors_and_size_query(lib):
    rc, need0 = _attn_variant("pkv_paged_attn_shared_prefix", lib, (), (0,))
    assert rc == 5 and need0 == _attn(lib)[1]           # no prefix: the plain call's workspace
    rc, need2 = _attn_variant("pkv_paged_attn_shared_prefix", lib, (), (2,))
    assert rc == 5 and need2 > need0                    # room for the prefix ranges' partials
    assert _attn_variant("pkv_paged_attn_shared_prefix", lib, (), (5,))[0] == 2    # beyond the table width
    assert _attn_variant("pkv_paged_attn_shared_prefix", lib, (), (-1,))[0] == 2
    f = ctypes.c_float
    rc, need8 = _attn_variant("pkv_paged_attn_shared_prefix_fp8", lib, (f(0.02), f(0.03)), (2,))
    assert rc == 5 and need8 == need2
    assert _attn_variant("pkv_paged_attn_shared_prefix_fp8", lib, (f(0.0), f(0.03)), (2,))[0] == 2


def test_copy_blocks_argument_errors(lib):
    P = ctypes.c_void_p
    fake, m = P(0x10000), P(0x20000)
    assert lib.pkv_copy_blocks(fake, 4, 2, 96, 16, m, 1, None, None) == 3
    assert lib.pkv_copy_blocks(fake, 4, 2, 128, 32, m, 1, None, None) == 3
    assert lib.pkv_copy_blocks(fake, 4, 0, 128, 16, m, 1, None, None) == 2
    assert lib.pkv_copy_blocks(fake, 4, 2, 128, 16, m, -1, None, None) == 2
    assert lib.pkv_copy_blocks(None, 4, 2, 128, 16, m, 1, None, None) == 1
    assert lib.pkv_copy_blocks(P(0x10008), 4, 2, 128, 16, m, 1, None, None) == 4
    assert lib.pkv_copy_blocks(fake, 4, 2, 128, 16, P(0x20004), 1, None, None) == 4
    assert lib.pkv_copy_blocks(fake, 4, 2, 128, 16, m, 0, None, None) == 0


def test_noalloc_refuses_before_any_launch(lib):
    P = ctypes.c_void_p
    f = ctypes.c_float

    def call(S, T, maxs, maxb, d=128):
        return lib.pkv_paged_attn_noalloc(P(0x10000), P(0x10000), 32 * d, P(0x10000), 1 << 20, P(0x20000), maxb,
                                          P(0x20000), P(0x20000), S, T, 1, maxs, 32, 8, d, 16, f(0.125), 0,
                                          None, None)
    assert call(2, 2, 64, 4, d=96) == 3                       # an argument error, as pkv_paged_attn
    assert call(0, 0, 64, 4) == 0                             # nothing to do
    # a batch whose scratch exceeds the fixed 256 MiB array is refused
    big = pkv.paged_attn_workspace_size(60000, 60000, 1, 65536, 32, 8, 128)
    assert big > (256 << 20)
    assert call(60000, 60000, 65536, 4096) == 5

"""The allocation-free entry point, pkv_paged_attn_noalloc.

It serves callers that cannot allocate GPU memory where they run attention
(code under a strict no-allocation policy, or a plugin whose host engine
hands it only inputs and outputs): instead of a caller
workspace it uses a fixed scratch array inside the library.  These tests
call it through the C ABI and compare it with the workspace path
(pkv_paged_attn + pkv_paged_attn_combine) on the same inputs, on two calls
in a row, within the attention tolerance of the other GPU tests, and with
the fp64 oracle directly; they also check that an error the GPU finds
reaches the caller's status word and that a clean call after it is clean.
The file is named to be collected last.
"""

import ctypes

import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from paged_kv_cache_111_gb300 import _build
from tolerance import ATOL, RTOL, check_close

pytestmark = pytest.mark.gpu

NOALLOC_MAX = 256 << 20        # PKV_NOALLOC_SCRATCH_BYTES in include/pkv.h


def _lib():
    _build.build()
    lib = pkv.load()
    fn = lib.pkv_paged_attn_noalloc
    P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    fn.argtypes = [P, P, i64, P, i64, P, i32, P, P, i32, i32, i32, i32, i32, i32, i32, i32, ctypes.c_float, i32,
                   P, P]
    fn.restype = ctypes.c_int
    return lib


def _setup(step):
    dev = {f: getattr(step, f).cuda().contiguous() for f in
           ("seq_lens", "query_start_loc", "block_tables", "query", "key", "value", "slot_mapping",
            "hist_key", "hist_value", "hist_slot_mapping")}
    pool = wl.make_poisoned_pool_like(step, device="cuda")
    pkv.kv_write(pool, dev["hist_key"], dev["hist_value"], dev["hist_slot_mapping"])
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    return dev, pool


def _call_noalloc(lib, step, dev, pool, out, status, num_splits=0, block_tables=None):
    bt = dev["block_tables"] if block_tables is None else block_tables
    return lib.pkv_paged_attn_noalloc(
        out.data_ptr(), dev["query"].data_ptr(), dev["query"].stride(0), pool.data_ptr(), step.num_blocks,
        bt.data_ptr(), step.max_blocks_per_seq, dev["seq_lens"].data_ptr(),
        dev["query_start_loc"].data_ptr(), step.num_seqs, step.num_tokens, step.max_query_len, step.max_seq_len,
        step.num_q_heads, step.num_kv_heads, step.head_size, step.block_size, ctypes.c_float(step.scale),
        num_splits, status.data_ptr(), torch.cuda.current_stream().cuda_stream)


def _workspace_path(step, dev, pool, num_splits=0):
    n = pkv.paged_attn_workspace_size(step.num_seqs, step.num_tokens, step.max_query_len, step.max_seq_len,
                                      step.num_q_heads, step.num_kv_heads, step.head_size)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.empty(step.num_tokens, step.num_q_heads, step.head_size, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn(out, dev["query"], pool, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                   step.max_query_len, step.max_seq_len, step.scale, ws, num_splits=num_splits)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    return out


def _close(a, b):
    a64, b64 = a.double(), b.double()
    assert torch.isfinite(a64).all()
    assert ((a64 - b64).abs() <= ATOL + RTOL * b64.abs()).all()


@pytest.mark.parametrize("num_splits", [0, 3])
def test_noalloc_matches_workspace_path_on_two_calls_in_a_row(num_splits):
    lib = _lib()
    # decodes split along their keys plus a prefill chunk starting mid-block
    step = wl.build_step("noalloc", [wl.RequestSpec(700, 1), wl.RequestSpec(33, 1), wl.RequestSpec(9, 40),
                                     wl.RequestSpec(1500, 1)], 16, 2, 128, 256, 77)
    dev, pool = _setup(step)
    ref = _workspace_path(step, dev, pool, num_splits)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(lib, step, dev, pool, out, status, num_splits) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _close(out, ref)


def test_noalloc_second_call_with_other_sizes_overwrites_the_scratch():
    lib = _lib()
    a = wl.build_step("a", [wl.RequestSpec(400, 1), wl.RequestSpec(64, 1)], 8, 8, 64, 64, 5)
    b = wl.build_step("b", [wl.RequestSpec(90, 2), wl.RequestSpec(0, 30), wl.RequestSpec(260, 1)], 8, 2, 128, 64, 6)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in (a, b):
        dev, pool = _setup(step)
        ref = _workspace_path(step, dev, pool)
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(lib, step, dev, pool, out, status) == 0
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _close(out, ref)


def test_noalloc_refuses_sizes_beyond_its_scratch():
    lib = _lib()
    # workspace for 1M single-token requests of 4096 tokens: far above the scratch
    need = pkv.paged_attn_workspace_size(1 << 20, 1 << 20, 1, 4096, 32, 32, 128)
    assert need > NOALLOC_MAX
    fake = ctypes.c_void_p(1 << 20)              # never dereferenced: refused before any launch
    rc = lib.pkv_paged_attn_noalloc(fake, fake, 32 * 128, fake, 1 << 20, fake, 256, fake, fake, 1 << 20, 1 << 20,
                                    1, 4096, 32, 32, 128, 16, ctypes.c_float(0.1), 0, None, None)
    assert rc == 5                                # PKV_ERR_WORKSPACE


@pytest.mark.parametrize("kind", ["decode only", "mixed with a chunk"])
def test_noalloc_matches_the_oracle(kind):
    lib = _lib()
    if kind == "decode only":
        step = wl.build_step("noalloc-decode", [wl.RequestSpec(c, 1) for c in (0, 15, 16, 300, 1100, 2047)],
                             32, 4, 64, 512, 91)
    else:
        step = wl.build_step("noalloc-mixed", [wl.RequestSpec(700, 1), wl.RequestSpec(0, 200),
                                               wl.RequestSpec(45, 3), wl.RequestSpec(1500, 1)], 32, 8, 128, 512, 92)
    dev, pool = _setup(step)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.full((step.num_tokens, step.num_q_heads, step.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    assert _call_noalloc(lib, step, dev, pool, out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, f"noalloc {kind}")


def test_noalloc_forwards_a_device_error_then_a_clean_call_is_clean():
    lib = _lib()
    step = wl.build_step("noalloc-err", [wl.RequestSpec(40, 1), wl.RequestSpec(10, 1)], 4, 2, 64, 64, 11)
    dev, pool = _setup(step)
    # a block id outside the pool: loaded as zeros by the bounded TMA, reported
    bad = dev["block_tables"].clone()
    bad[0, 1] = step.num_blocks + 1000
    out = torch.zeros(step.num_tokens, 4, 64, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert _call_noalloc(lib, step, dev, pool, out, status, block_tables=bad) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 7                # PKV_ERR_DEVICE_INDEX
    # the word keeps the first error: a clean call does not clear it
    assert _call_noalloc(lib, step, dev, pool, out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 7
    # a clean call into a cleared word: the shared scratch carries no stale status
    status.zero_()
    out.fill_(float("nan"))
    assert _call_noalloc(lib, step, dev, pool, out, status) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, "noalloc after an error")
    # an earlier error in the caller's word (say, from the cache write) is kept
    status.fill_(8)
    assert _call_noalloc(lib, step, dev, pool, out, status, block_tables=bad) == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 8

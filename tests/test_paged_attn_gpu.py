"""paged_attn + paged_attn_combine on the GPU against the fp64 oracle.

Tolerance |gpu - ref| <= 2e-3 + 1e-2 |ref| elementwise (tests/tolerance.py).
"""

import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import attend, new_pool, run_step, to_dev, workspace_for, write_history
from tolerance import check_close

pytestmark = pytest.mark.gpu


def custom(reqs, H, Hkv, d, seed=1, nb=None, **kw):
    specs = [wl.RequestSpec(c, q) for c, q in reqs]
    need = sum((c + q + 15) // 16 for c, q in reqs) + 8
    return wl.build_step("custom", specs, H, Hkv, d, nb or max(2 * need, 16), seed, **kw)


def compare(step, num_splits=0, what=""):
    _, out, status = run_step(step, num_splits=num_splits)
    assert status == 0, pkv.STATUS_NAMES.get(status, status)
    _, ref, _ = oracle.run_step(step)
    return check_close(out, ref, what or step.name)


@pytest.mark.parametrize("name", ["tiny-decode", "tinyllama-decode", "llama3-8b-mixed", "llama3-70b-prefix"])
def test_named_workloads_full_size(name):
    compare(wl.make_workload(name))


def test_llama13b_full_size_every_row():
    """The 13B batch (256 requests, 100000-block cache) runs whole on the GPU,
    and every one of its output rows is checked against the oracle.  The
    oracle runs on the same batch with its pool compacted to the blocks the
    tables use (about 4 GB on the host); each request sees the same keys,
    values and queries, so the rows compare one to one."""
    step = wl.make_workload("llama13b-decode")
    _, out, status = run_step(step)
    assert status == 0
    out = out.cpu()
    sub = step.subset(range(step.num_seqs))
    assert torch.equal(sub.query, step.query)
    _, ref, _ = oracle.run_step(sub)
    check_close(out, ref, "llama13b every row")


EDGE = [
    # seq_len edges around the 16-token page: 1, 15, 16, 17, 31, 32, 33
    ("page edges mha d64", [(0, 1), (14, 1), (15, 1), (16, 1), (30, 1), (31, 1), (32, 1)], 4, 4, 64),
    ("page edges gqa8 d128", [(0, 1), (14, 1), (15, 1), (16, 1), (30, 1), (31, 1), (32, 1)], 16, 2, 128),
    ("chunk mid-block + ragged", [(5, 40), (17, 1), (0, 17), (33, 3)], 8, 2, 128),
    ("multi-token decode rows", [(40, 2), (100, 3), (7, 4), (63, 2)], 16, 2, 64),
    ("gqa4 tile spans queries", [(20, 5), (0, 9), (48, 4)], 8, 2, 128),
    ("mqa G=32", [(70, 1), (3, 2), (0, 5)], 32, 1, 64),
    ("G=16 one tile per token", [(90, 1), (31, 1)], 32, 2, 128),
    ("empty requests", [(20, 4), (0, 0), (47, 1), (5, 0)], 8, 4, 64),
    ("long prefill chunk", [(130, 300), (0, 1)], 8, 2, 128),
    # decode tiles of exactly 8 rows (q_r * G = 8) holding several query tokens each
    ("8-row tiles q=4 G=2", [(50, 4), (3, 4), (200, 2), (17, 1)], 4, 2, 64),
    ("8-row tiles q=2 G=4 split keys", [(900, 2), (30, 2), (0, 1)], 16, 4, 128),
]


@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
def test_edge_cases(case):
    name, reqs, H, Hkv, d = case
    compare(custom(reqs, H, Hkv, d, seed=zlib.crc32(name.encode()) % 1000), what=name)


PREFILL = [
    # requests whose rows (query tokens x GQA group) exceed 64 run on the tcgen05 prefill kernel
    ("mha d128 c=0 q=300", [(0, 300)], 4, 4, 128, None),
    ("gqa4 d128 long context", [(1000, 200), (17, 1)], 16, 4, 128, None),
    ("gqa8 d64 mid-block", [(37, 90), (200, 70)], 16, 2, 64, None),
    ("gqa2 d128 ragged tail", [(5, 129), (0, 33), (250, 1)], 8, 4, 128, None),
    ("mha d64 partial last page", [(100, 150)], 2, 2, 64, None),
    ("gqa16 d128", [(64, 40), (3, 10)], 32, 2, 128, None),
    ("peaked softmax (scale 1.0)", [(300, 260), (50, 1)], 8, 2, 128, 1.0),
    ("long chunk 4096 context", [(4096, 256)], 8, 1, 128, None),
]


@pytest.mark.parametrize("case", PREFILL, ids=[c[0] for c in PREFILL])
def test_prefill_tensor_core_path(case):
    name, reqs, H, Hkv, d, scale = case
    step = custom(reqs, H, Hkv, d, seed=zlib.crc32(name.encode()) % 1000, scale=scale)
    compare(step, what=name)


def test_more_requests_than_the_plan_stages():
    # 1500 requests (the plan keeps up to 1024 in shared memory; beyond that
    # its per-request state lives in the workspace): decode rows, short
    # multi-token rows, one long chunk on the tensor-core kernel, empty requests
    rng = np.random.default_rng(11)
    reqs = [(int(rng.integers(0, 160)), 1) for _ in range(1500)]
    for i in range(0, 1500, 97):
        reqs[i] = (int(rng.integers(0, 60)), int(rng.integers(2, 5)))
    reqs[5] = (40, 0)
    reqs[700] = (0, 0)
    reqs[1499] = (33, 90)
    compare(custom(reqs, 8, 2, 64, seed=11), what="1500 requests")


@pytest.mark.parametrize("splits", [1, 2, 3, 7, 32])
def test_forced_split_counts_merge_to_the_same_result(splits):
    step = custom([(700, 1), (33, 1), (1500, 1), (0, 1), (255, 1)], 16, 2, 128, seed=splits)
    compare(step, num_splits=splits, what=f"splits={splits}")


def test_long_sequence_and_max_splits():
    step = custom([(32767, 1), (9000, 2)], 8, 1, 128, seed=5)
    compare(step, what="32k context")


def test_shared_prefix_and_cow_forks():
    step = custom([(200, 1), (260, 1), (143, 1), (64, 1)], 16, 2, 128, seed=8, shared_prefix_len=64,
                  forks=[0, 1, 3])
    compare(step, what="prefix+forks")


def test_relabelled_blocks_give_bit_identical_output():
    step = custom([(300, 1), (45, 1), (1000, 1)], 8, 8, 128, seed=9)
    _, out1, _ = run_step(step)
    # relabel every physical block by a permutation (inputs only)
    perm = torch.randperm(step.num_blocks, generator=torch.Generator().manual_seed(2))
    B = 16

    def rl(slots):
        return torch.where(slots >= 0, perm[torch.div(slots, B, rounding_mode="floor").clamp(min=0)] * B + slots % B,
                           slots)
    step2 = wl.Step(**{**step.__dict__})
    step2.block_tables = torch.where(step.block_tables >= 0, perm[step.block_tables.long().clamp(min=0)].int(),
                                     step.block_tables)
    step2.slot_mapping = rl(step.slot_mapping)
    step2.hist_slot_mapping = rl(step.hist_slot_mapping)
    _, out2, _ = run_step(step2)
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


def test_nan_poisoned_tail_slots_do_not_leak():
    # every request ends mid-page: slots past seq_len hold NaN in the pool
    step = custom([(4, 1), (20, 1), (37, 3), (2, 12)], 8, 2, 64, seed=10)
    compare(step, what="nan tails")


def test_device_errors_are_reported_without_a_fault():
    step = custom([(40, 1), (10, 1)], 4, 2, 64, seed=11)
    dev = to_dev(step)
    pool = new_pool(step)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    ws = workspace_for(step)
    # a block id outside the pool: loaded as zeros by the bounded TMA, reported
    bt = dev["block_tables"].clone()
    bt[0, 1] = step.num_blocks + 1000
    out = torch.zeros(step.num_tokens, 4, 64, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn(out, dev["query"], pool, bt, dev["seq_lens"], dev["query_start_loc"],
                   step.max_query_len, step.max_seq_len, step.scale, ws)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 7          # PKV_ERR_DEVICE_INDEX
    # a seq_len above the host hint: that request is refused, reported
    sl = dev["seq_lens"].clone()
    sl[1] = step.max_seq_len + 1
    out.zero_()
    pkv.paged_attn(out, dev["query"], pool, dev["block_tables"], sl, dev["query_start_loc"],
                   step.max_query_len, step.max_seq_len, step.scale, ws)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 8          # PKV_ERR_DEVICE_METADATA
    assert (out[1] == 0).all()
    # combine with sizes that do not match the workspace's last paged_attn
    pkv.paged_attn(out, dev["query"], pool, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                   step.max_query_len, step.max_seq_len, step.scale, ws)
    other = torch.zeros(step.num_tokens + 1, 4, 64, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn_combine(other, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 10         # PKV_ERR_PROTOCOL
    assert (other == 0).all()


def test_out_of_pool_block_in_a_tensor_core_chunk_is_reported():
    """A block id past the pool in a chunk on the tensor-core kernel loads as
    zeros (the TMA box lies outside the tensor map) and is reported; the other
    request's row is unaffected."""
    step = custom([(40, 1), (10, 150)], 8, 2, 128, seed=12)          # request 1: 600 rows, tcgen05 tiles
    dev = to_dev(step)
    pool = new_pool(step)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    ws = workspace_for(step)
    bt = dev["block_tables"].clone()
    bt[1, 3] = step.num_blocks + 1000
    out = torch.zeros(step.num_tokens, 8, 128, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn(out, dev["query"], pool, bt, dev["seq_lens"], dev["query_start_loc"],
                   step.max_query_len, step.max_seq_len, step.scale, ws)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 7          # PKV_ERR_DEVICE_INDEX
    _, ref, _ = oracle.run_step(step.subset([0]))
    check_close(out[:1], ref, "request beside the bad chunk")


def test_workspace_query_and_too_small_workspace():
    step = custom([(40, 1)], 4, 2, 64, seed=12)
    need = pkv.paged_attn_workspace_size(1, 1, 1, 41, 4, 2, 64)
    assert need > 256
    dev = to_dev(step)
    pool = new_pool(step)
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    out = torch.zeros(1, 4, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PagedKVError) as e:
        pkv.paged_attn(out, dev["query"], pool, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                       1, 41, step.scale, small)
    assert e.value.code == 5
    torch.cuda.synchronize()
    assert (out == 0).all()


def test_empty_batch():
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    pool = torch.zeros(4, 2, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    q = torch.zeros(0, 4, 64, dtype=torch.bfloat16, device="cuda")
    e32 = torch.zeros(0, dtype=torch.int32, device="cuda")
    pkv.paged_attn(out, q, pool, torch.zeros(0, 1, dtype=torch.int32, device="cuda"), e32,
                   torch.zeros(1, dtype=torch.int32, device="cuda"), 0, 0, 0.125, ws)
    pkv.paged_attn_combine(out, ws)
    pkv.kv_write(pool, q[:, :2], q[:, :2], torch.zeros(0, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()


def test_same_workspace_reused_in_stream_order():
    a = custom([(100, 1), (300, 1)], 8, 2, 128, seed=13)
    dev = to_dev(a)
    pool = new_pool(a)
    write_history(a, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    ws = workspace_for(a)
    o1 = attend(a, pool, dev, ws)
    o2 = attend(a, pool, dev, ws, num_splits=5)
    torch.cuda.synchronize()
    _, ref, _ = oracle.run_step(a)
    check_close(o1, ref, "first")
    check_close(o2, ref, "second")

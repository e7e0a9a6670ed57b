"""Decode-only calls that the decode kernel plans itself, against the fp64 oracle.

A small batch of split rows (every request's q_r * G <= 16, automatic splits,
few enough (request, kv head) pairs and pages for the decode grid) runs with
no plan kernel: with at most 64 requests every warp of a chunk CTA plans the
call by itself in registers, with more every decode CTA plans it in shared
memory, and the grid's last CTA writes the header and the split tokens for
the combine.  A
forced split count, a shared-prefix call or a large batch goes through the
plan kernel instead.  Either way the rows must match the oracle; the status
word must report a bad block id, bad lengths, and clear on the next clean call.
"""

import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import attend, new_pool, run_step, to_dev, workspace_for, write_history
from tolerance import check_close

pytestmark = pytest.mark.gpu


def custom(reqs, H, Hkv, d, seed=1):
    specs = [wl.RequestSpec(c, q) for c, q in reqs]
    need = sum((c + q + 15) // 16 for c, q in reqs) + 8
    return wl.build_step("self-plan", specs, H, Hkv, d, max(2 * need, 16), seed)


@pytest.mark.parametrize("num_splits", [0, 3])
def test_the_same_batch_with_and_without_the_plan_kernel(num_splits):
    """num_splits = 0 lets the decode kernel plan; 3 forces the plan kernel."""
    gen = torch.Generator().manual_seed(41)
    lens = torch.randint(1, 900, (40,), generator=gen).tolist()
    step = custom([(l - 1, 1) for l in lens], 16, 4, 64, seed=41)
    _, out, status = run_step(step, num_splits=num_splits)
    assert status == 0, pkv.STATUS_NAMES.get(status, status)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, f"num_splits={num_splits}")


@pytest.mark.parametrize("n,H,Hkv,d,q", [
    (1, 8, 8, 128, 1),       # one request: a grid of one chunk CTA and the header CTA
    (3, 32, 8, 128, 2),      # two query tokens per row group (G = 4, 8 rows)
    (16, 40, 40, 128, 1),    # MHA
    (64, 8, 2, 64, 1),       # the most requests every warp plans by itself (two per lane)
    (65, 8, 2, 64, 1),       # one more: the chunk CTAs plan in shared memory
    (300, 8, 2, 64, 1),
    (1100, 8, 2, 64, 1),     # more requests than the decode kernel plans itself: the plan kernel
])
def test_batches_on_both_sides_of_the_self_plan_bound(n, H, Hkv, d, q):
    gen = torch.Generator().manual_seed(n)
    lens = torch.randint(q, 400, (n,), generator=gen).tolist()
    step = custom([(l - q, q) for l in lens], H, Hkv, d, seed=n)
    _, out, status = run_step(step)
    assert status == 0, pkv.STATUS_NAMES.get(status, status)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, f"{n} requests")


def test_errors_of_a_self_planned_call_then_a_clean_call():
    step = custom([(100, 1), (37, 1), (250, 1)], 8, 2, 64, seed=7)
    dev = to_dev(step)
    pool = new_pool(step)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    ws = workspace_for(step)
    _, ref, _ = oracle.run_step(step)
    # a block id past the pool in request 2's table: reported, the others' rows intact
    bt = dev["block_tables"].clone()
    bt[2, 3] = step.num_blocks + 7
    out = attend(step, pool, dict(dev, block_tables=bt), ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 7            # PKV_ERR_DEVICE_INDEX
    check_close(out[:2], ref[:2], "rows beside the bad block")
    # a length above the host bound: refused and reported
    sl = dev["seq_lens"].clone()
    sl[0] = step.max_seq_len + 1
    attend(step, pool, dict(dev, seq_lens=sl), ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 8            # PKV_ERR_DEVICE_METADATA
    # the next clean call in the same workspace reports nothing and matches the oracle
    out = attend(step, pool, dev, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    check_close(out, ref, "clean call after errors")


def test_repeated_self_planned_calls_in_stream_order():
    """Each call's header and status are written by its own last CTA while the
    previous call's combine may still be reading the workspace's split rows."""
    a = custom([(60, 1), (500, 1), (9, 1), (200, 1)], 16, 4, 128, seed=3)
    b = custom([(300, 1), (20, 1)], 16, 4, 128, seed=4)
    ra = oracle.run_step(a)[1]
    rb = oracle.run_step(b)[1]
    pools = []
    for st in (a, b):
        dev = to_dev(st)
        pool = new_pool(st)
        write_history(st, pool, dev)
        pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
        pools.append((pool, dev))
    n = max(pkv.paged_attn_workspace_size(s.num_seqs, s.num_tokens, s.max_query_len, s.max_seq_len,
                                          s.num_q_heads, s.num_kv_heads, s.head_size) for s in (a, b))
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    outs = []
    for i in range(6):
        st = (a, b)[i % 2]
        pool, dev = pools[i % 2]
        outs.append(attend(st, pool, dev, ws))
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    for i, o in enumerate(outs):
        check_close(o, (ra, rb)[i % 2], f"call {i}")

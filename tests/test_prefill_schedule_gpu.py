"""The persistent tensor-core prefill kernel's dynamic schedule.

One CTA per SM takes work items (a 128-row tile for one kv head) from a
counter the plan zeroes, largest first; each CTA records how many items it
took.  Every item is taken exactly once (the outputs are checked against the
oracle by the attention tests; here the count is), each CTA of the grid takes
at least one, and a step without prefill tiles leaves the record zeroed.
"""

import pytest
import torch

import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import new_pool, to_dev, workspace_for, write_history

pytestmark = pytest.mark.gpu

DECODE_TILE_MAX_ROWS = 64      # rows above this go to the tensor-core prefill kernel
ITEM_ROWS = 128                # rows of one work item of that kernel


def prefill_items(step):
    G = step.num_q_heads // step.num_kv_heads
    n = 0
    for r in range(step.num_seqs):
        rows = (int(step.query_start_loc[r + 1]) - int(step.query_start_loc[r])) * G
        if rows > DECODE_TILE_MAX_ROWS:
            n += -(-rows // ITEM_ROWS) * step.num_kv_heads
    return n


def attend(step, ws=None):
    dev = to_dev(step)
    pool = new_pool(step)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    ws = workspace_for(step) if ws is None else ws
    out = torch.empty(step.num_tokens, step.num_q_heads, step.head_size, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn(out, dev["query"], pool, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                   step.max_query_len, step.max_seq_len, step.scale, ws)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    return ws


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def test_every_item_of_the_mixed_step_is_taken_once():
    step = wl.make_workload("llama3-8b-mixed")
    items = prefill_items(step)
    assert items == 512
    pf, px = pkv.workspace_schedule(attend(step))
    assert sum(pf) == items
    assert len(pf) == min(sm_count(), items)
    assert min(pf) >= 1 and px == []


@pytest.mark.parametrize("reqs,H,Hkv,d", [
    ([(0, 300)], 4, 4, 128),                 # fewer items than SMs: one each
    ([(1000, 200), (17, 1), (5, 129)], 16, 4, 128),
    ([(37, 90), (200, 70), (0, 600)], 16, 2, 64),
])
def test_item_counts_on_custom_steps(reqs, H, Hkv, d):
    specs = [wl.RequestSpec(c, q) for c, q in reqs]
    need = sum((c + q + 15) // 16 for c, q in reqs) + 8
    step = wl.build_step("sched", specs, H, Hkv, d, 2 * need, 9)
    items = prefill_items(step)
    pf, _ = pkv.workspace_schedule(attend(step))
    assert sum(pf) == items
    assert len(pf) == min(sm_count(), items)
    assert min(pf) >= 1


def test_a_step_without_prefill_tiles_leaves_the_record_zeroed():
    big = wl.make_workload("llama3-8b-mixed")
    ws = torch.zeros(1 << 26, dtype=torch.uint8, device="cuda")
    pf, _ = pkv.workspace_schedule(attend(big, ws))
    assert sum(pf) == prefill_items(big)
    small = wl.make_workload("tiny-decode")
    pf, px = pkv.workspace_schedule(attend(small, ws))
    assert pf == [] and px == []

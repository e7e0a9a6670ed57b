"""Cascade attention over a shared table prefix against the oracle.

pkv_paged_attn_shared_prefix computes the same result as pkv_paged_attn: the
keys of the shared blocks are attended once per kv head by every sharing row
(tensor-core tiles) and merged with each row's own keys by the log-sum-exp
combine.  Requests that do not share the prefix (or whose context does not
cover it, or whose rows exceed one decode tile) take the ordinary path.
"""

import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import new_pool, to_dev, write_history
from tolerance import check_close

pytestmark = pytest.mark.gpu


_last_workspace = [None]


def run_cascade(step, prefix_blocks, num_splits=0):
    dev = to_dev(step)
    pool = new_pool(step)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    n = pkv.paged_attn_shared_prefix_workspace_size(step.num_seqs, step.num_tokens, step.max_query_len,
                                                    step.max_seq_len, step.num_q_heads, step.num_kv_heads,
                                                    step.head_size, prefix_blocks)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.full((step.num_tokens, step.num_q_heads, step.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    pkv.paged_attn_shared_prefix(out, dev["query"], pool, dev["block_tables"], dev["seq_lens"],
                                 dev["query_start_loc"], step.max_query_len, step.max_seq_len, step.scale,
                                 prefix_blocks, ws, num_splits=num_splits)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    _last_workspace[0] = ws
    return out


def test_prefix_sharing_workload_full_size():
    step = wl.make_workload("llama3-70b-prefix")
    out = run_cascade(step, 64)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, "70b prefix cascade")


CASES = [
    # (requests (context, query), H, Hkv, d, shared prefix tokens, forks, prefix blocks passed)
    ("gqa8 d128 with forks", [(300, 1), (257, 1), (130, 1), (64, 1)], 16, 2, 128, 64, [0, 2], 4),
    ("prefix not a tile multiple", [(200, 1), (180, 1), (90, 1)], 8, 2, 128, 80, [], 5),
    ("d64 mha", [(150, 1), (99, 1), (64, 1)], 4, 4, 64, 48, [1], 3),
    ("multi-token rows", [(120, 2), (70, 2), (66, 1)], 16, 2, 128, 64, [], 4),
    ("passing fewer blocks than shared", [(300, 1), (200, 1)], 16, 2, 128, 128, [], 3),
    # G = 3 does not divide a 128-row tile: the call falls back to the plain path
    ("group of three, no tensor-core tile", [(200, 1), (150, 1)], 6, 2, 128, 64, [], 4),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_cascade_cases(case):
    name, reqs, H, Hkv, d, shared, forks, K = case
    specs = [wl.RequestSpec(c, q) for c, q in reqs]
    step = wl.build_step("casc", specs, H, Hkv, d, 512, 61, shared_prefix_len=shared, forks=forks)
    out = run_cascade(step, K)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, name)


def test_mixed_batch_with_non_sharers_a_chunk_and_short_contexts():
    # requests 0-2 share 4 blocks; request 3 has its own table; request 4's
    # context is shorter than the prefix; request 5 is a prefill chunk
    specs = [wl.RequestSpec(150, 1), wl.RequestSpec(90, 1), wl.RequestSpec(70, 1), wl.RequestSpec(200, 1),
             wl.RequestSpec(66, 1), wl.RequestSpec(64, 80)]
    step = wl.build_step("mixed", specs, 16, 4, 128, 512, 62, shared_prefix_len=64,
                         shared_prefix_requests=[0, 1, 2, 4, 5])
    out = run_cascade(step, 4)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, "mixed cascade batch")


def test_request_zero_not_sharing_means_no_cascade():
    specs = [wl.RequestSpec(100, 1), wl.RequestSpec(150, 1), wl.RequestSpec(140, 1)]
    step = wl.build_step("nozero", specs, 16, 2, 128, 256, 64, shared_prefix_len=64, shared_prefix_requests=[1, 2])
    out = run_cascade(step, 4)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, "request 0 not sharing")


@pytest.mark.parametrize("splits", [1, 3, 32])
def test_cascade_with_forced_suffix_splits(splits):
    # 1024-token prefix (8 KV tiles, cut into ranges) and suffixes of up to 60 pages
    specs = [wl.RequestSpec(2000, 1), wl.RequestSpec(1300, 1), wl.RequestSpec(1025, 1)]
    step = wl.build_step("split", specs, 8, 1, 128, 512, 63, shared_prefix_len=1024)
    out = run_cascade(step, 64, num_splits=splits)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, f"cascade splits={splits}")


def test_cascade_pass_with_more_items_than_ctas():
    # 1024 sharers with 1 or 2 query tokens x G = 8: 12288 rows per kv head,
    # 96 row tiles x 4 kv heads = 384 cascade items (one prefix range), more
    # than one per persistent CTA
    rng = torch.Generator().manual_seed(65)
    ctx = (256 + torch.randint(0, 48, (1024,), generator=rng)).tolist()
    q = (1 + (torch.arange(1024) % 2)).tolist()
    specs = [wl.RequestSpec(int(c), int(n)) for c, n in zip(ctx, q)]
    step = wl.build_step("many", specs, 32, 4, 128, 8192, 65, shared_prefix_len=256)
    out = run_cascade(step, 16)
    _, px = pkv.workspace_schedule(_last_workspace[0])
    assert sum(px) == 384 and len(px) == min(384, torch.cuda.get_device_properties(0).multi_processor_count)
    assert min(px) >= 1
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, "cascade, 384 items")


def test_cascade_with_more_requests_than_the_plan_stages():
    # 1100 sharers of a 64-token prefix: the plan compares every table with
    # request 0's and keeps the per-request state in the workspace
    rng = torch.Generator().manual_seed(66)
    ctx = (64 + torch.randint(0, 40, (1100,), generator=rng)).tolist()
    specs = [wl.RequestSpec(int(c), 1) for c in ctx]
    step = wl.build_step("many", specs, 16, 2, 64, 8192, 66, shared_prefix_len=64)
    out = run_cascade(step, 4)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, "cascade, 1100 sharers")

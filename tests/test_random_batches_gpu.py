"""Seeded random batches through the whole GPU path against the fp64 oracle.

Each case draws a head layout (MHA, GQA 2/4/8, MQA), a head size, a number
of requests, and per request a context and a query length from a mix of
decode rows, short multi-token rows, chunks that land on the decode kernel's
16-row tiles and chunks long enough for the tensor-core kernel, plus empty
requests.  Some cases force a split count, some use a shared table prefix
with the cascade call, some an E4M3 cache.  Every row is compared with the
oracle within |gpu - ref| <= 2e-3 + 1e-2 |ref|.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import run_step, to_dev
from tolerance import check_close

pytestmark = pytest.mark.gpu

LAYOUTS = [(4, 4), (8, 4), (16, 4), (32, 4), (8, 1), (16, 16)]
QUERY_LENS = [0, 1, 1, 1, 1, 2, 3, 4, 9, 17, 40, 70, 130]


def draw_case(seed: int):
    rng = np.random.default_rng(1000 + seed)
    H, Hkv = LAYOUTS[int(rng.integers(len(LAYOUTS)))]
    d = int(rng.choice([64, 128]))
    S = int(rng.integers(1, 10))
    reqs = []
    for _ in range(S):
        q = int(rng.choice(QUERY_LENS))
        c = int(rng.integers(0, 400)) if rng.random() < 0.8 else int(rng.integers(0, 20))
        reqs.append((c, q))
    if all(q == 0 for _, q in reqs):
        reqs[0] = (reqs[0][0], 1)
    splits = int(rng.choice([0, 0, 0, 1, 3, 32]))
    scale = None if rng.random() < 0.7 else float(rng.choice([0.05, 0.3, 1.0]))
    return reqs, H, Hkv, d, splits, scale


def build(reqs, H, Hkv, d, seed, scale, **kw):
    specs = [wl.RequestSpec(c, q) for c, q in reqs]
    need = sum((c + q + 15) // 16 for c, q in reqs) + 8
    return wl.build_step("random", specs, H, Hkv, d, max(2 * need, 16), seed, scale=scale, **kw)


@pytest.mark.parametrize("seed", range(24))
def test_random_batch(seed):
    reqs, H, Hkv, d, splits, scale = draw_case(seed)
    step = build(reqs, H, Hkv, d, seed, scale)
    _, out, status = run_step(step, num_splits=splits)
    assert status == 0, pkv.STATUS_NAMES.get(status, status)
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, f"random batch {seed}: {reqs} H={H} Hkv={Hkv} d={d} splits={splits}")


@pytest.mark.parametrize("seed", range(8))
def test_random_batch_with_shared_prefix(seed):
    rng = np.random.default_rng(2000 + seed)
    H, Hkv = LAYOUTS[int(rng.integers(len(LAYOUTS)))]
    d = int(rng.choice([64, 128]))
    prefix_blocks = int(rng.integers(1, 9))
    S = int(rng.integers(2, 12))
    # every request's context covers the shared prefix; a few rows per request
    reqs = [(prefix_blocks * 16 + int(rng.integers(0, 200)), int(rng.choice([1, 1, 2]))) for _ in range(S)]
    step = build(reqs, H, Hkv, d, 50 + seed, None, shared_prefix_len=prefix_blocks * 16)
    dev = to_dev(step)
    pool = wl.make_poisoned_pool_like(step, device="cuda")
    for a in range(0, dev["hist_slot_mapping"].shape[0], 1 << 16):
        b = min(dev["hist_slot_mapping"].shape[0], a + (1 << 16))
        pkv.kv_write(pool, dev["hist_key"][a:b], dev["hist_value"][a:b], dev["hist_slot_mapping"][a:b])
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    n = pkv.paged_attn_shared_prefix_workspace_size(step.num_seqs, step.num_tokens, step.max_query_len,
                                                    step.max_seq_len, H, Hkv, d, prefix_blocks)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.full((step.num_tokens, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn_shared_prefix(out, dev["query"], pool, dev["block_tables"], dev["seq_lens"],
                                 dev["query_start_loc"], step.max_query_len, step.max_seq_len, step.scale,
                                 prefix_blocks, ws)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    _, ref, _ = oracle.run_step(step)
    check_close(out, ref, f"random cascade batch {seed}: {reqs} H={H} Hkv={Hkv} d={d} prefix={prefix_blocks}")


@pytest.mark.parametrize("seed", range(8))
def test_random_batch_fp8(seed):
    reqs, H, Hkv, d, splits, scale = draw_case(100 + seed)
    step = build(reqs, H, Hkv, d, 100 + seed, scale)
    rng = np.random.default_rng(3000 + seed)
    k_scale, v_scale = float(np.float32(rng.uniform(0.002, 0.05))), float(np.float32(rng.uniform(0.002, 0.05)))
    dev = to_dev(step)
    cache = torch.full(step.pool_shape(), 0x7F, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for a in range(0, dev["hist_slot_mapping"].shape[0], 1 << 16):
        b = min(dev["hist_slot_mapping"].shape[0], a + (1 << 16))
        pkv.kv_write_fp8(cache, dev["hist_key"][a:b], dev["hist_value"][a:b], dev["hist_slot_mapping"][a:b],
                         k_scale, v_scale, st)
    pkv.kv_write_fp8(cache, dev["key"], dev["value"], dev["slot_mapping"], k_scale, v_scale, st)
    n = pkv.paged_attn_workspace_size(step.num_seqs, step.num_tokens, step.max_query_len, step.max_seq_len,
                                      H, Hkv, d)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    out = torch.full((step.num_tokens, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn_fp8(out, dev["query"], cache, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                       step.max_query_len, step.max_seq_len, step.scale, k_scale, v_scale, ws, num_splits=splits)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and pkv.workspace_status(ws) == 0
    _, ref, _ = oracle.run_step_fp8(step, k_scale, v_scale)
    check_close(out, ref, f"random fp8 batch {seed}: {reqs} H={H} Hkv={Hkv} d={d} splits={splits}")

"""Pins for the CPU oracle: it is checked against things other than itself.

* torch's own scaled_dot_product_attention (fp64, CPU, grouped-query mode) on
  contiguous K/V built by the input generator, never read from a cache;
* the pages' worked examples (tests/golden/*.json, each with its citation);
* closed forms and invariants: a single key, two keys, uniform keys, zero
  scale, weights summing to one, relabelled physical blocks, shared prefix
  blocks against private copies, and the log-sum-exp merge of a split key
  range.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def bf16_to_f64(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float64)


def sdpa_reference(step: wl.Step):
    """torch SDPA (fp64) per request on contiguous K/V; returns [T, H, d] fp64."""
    out = torch.zeros(step.num_tokens, step.num_q_heads, step.head_size, dtype=torch.float64)
    for r in range(step.num_seqs):
        q0, q1 = int(step.query_start_loc[r]), int(step.query_start_loc[r + 1])
        if q1 == q0:
            continue
        L = int(step.seq_lens[r])
        c = L - (q1 - q0)
        k, v = step.request_kv(r)                      # [L, Hkv, d]
        q = bf16_to_f64(step.query[q0:q1]).permute(1, 0, 2).unsqueeze(0)   # [1, H, q, d]
        kk = bf16_to_f64(k).permute(1, 0, 2).unsqueeze(0)                 # [1, Hkv, L, d]
        vv = bf16_to_f64(v).permute(1, 0, 2).unsqueeze(0)
        i = torch.arange(q1 - q0).unsqueeze(1)
        j = torch.arange(L).unsqueeze(0)
        mask = j <= (c + i)                                                # [q, L]
        o = torch.nn.functional.scaled_dot_product_attention(
            q, kk, vv, attn_mask=mask, scale=step.scale, enable_gqa=True)
        out[q0:q1] = o[0].permute(1, 0, 2)
    return out


def custom(reqs, H, Hkv, d, nb=None, seed=1, **kw):
    specs = [wl.RequestSpec(c, q) for c, q in reqs]
    need = sum((c + q + 15) // 16 for c, q in reqs) + 4
    return wl.build_step("custom", specs, H, Hkv, d, nb or max(need * 2, 8), seed, **kw)


CASES = [
    # (requests as (context, query), H, Hkv, d)
    ([(0, 1), (14, 1), (15, 1), (16, 1), (30, 1), (31, 1), (32, 1)], 4, 4, 64),
    ([(17, 1), (40, 3), (5, 40), (0, 17)], 8, 2, 128),
    ([(100, 1), (0, 33), (16, 16), (33, 2)], 16, 2, 64),
    ([(63, 1), (9, 7), (0, 1)], 8, 8, 128),
    ([(20, 4), (0, 0), (47, 1)], 32, 4, 64),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_oracle_matches_torch_sdpa_on_contiguous_kv(case):
    reqs, H, Hkv, d = CASES[case]
    step = custom(reqs, H, Hkv, d, seed=100 + case)
    _, out, lse = oracle.run_step(step)
    ref = sdpa_reference(step).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_oracle_matches_sdpa_with_shared_prefix_and_forks():
    reqs = [(47, 1), (60, 1), (33, 1)]
    step = custom(reqs, 8, 2, 64, seed=7, shared_prefix_len=32, forks=[0, 2])
    assert step.num_seqs == 5
    _, out, _ = oracle.run_step(step)
    np.testing.assert_allclose(out, sdpa_reference(step).numpy(), rtol=1e-12, atol=1e-12)


def test_index_example_from_the_pages():
    g = golden("index_example.json")
    B = g["block_size"]
    assert B == wl.BLOCK_SIZE
    pos = g["token_position"]
    assert pos // B == g["logical_block"] and pos % B == g["offset"]
    assert g["block_table"][g["logical_block"]] == g["physical_block"]
    # the oracle's cache write puts slot 42*16+2 at physical block 42, offset 2
    d, hkv = 64, 1
    cache = oracle.new_cache(64, hkv, d)
    rng = np.random.default_rng(0)
    k = torch.from_numpy(rng.standard_normal((1, hkv, d)).astype(np.float32)).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((1, hkv, d)).astype(np.float32)).to(torch.bfloat16)
    slot = g["physical_block"] * B + g["offset"]
    oracle.kv_write(cache, k, v, torch.tensor([slot]))
    raw_k = k.view(torch.int16).numpy().view(np.uint16)
    raw_v = v.view(torch.int16).numpy().view(np.uint16)
    assert (cache[g["physical_block"], 0, 0, g["offset"]] == raw_k[0, 0]).all()
    assert (cache[g["physical_block"], 0, 1, g["offset"]] == raw_v[0, 0]).all()
    assert np.count_nonzero(cache != 0x7FC0) <= 2 * d
    # the oracle's read of logical token 18 through the table [17, 42] lands
    # on that slot: with a query that only key 18 matches strongly and a huge
    # scale, the output is that slot's value
    L = pos + 1
    table = torch.tensor([g["block_table"] + [-1]], dtype=torch.int32)
    kk = torch.zeros(L, hkv, d)
    kk[pos] = 1.0
    q = torch.zeros(1, 1, d)
    q[0, 0, :] = 1.0
    # keys 0..17 in block 17 and the first two slots of block 42 (zero keys),
    # key 18 is the written one at (42, 2) but with K = ones
    cache2 = oracle.new_cache(64, hkv, d)
    slots = [g["block_table"][j // B] * B + j % B for j in range(L)]
    vals = torch.from_numpy(rng.standard_normal((L, hkv, d)).astype(np.float32)).to(torch.bfloat16)
    oracle.kv_write(cache2, kk.to(torch.bfloat16), vals, torch.tensor(slots))
    out, lse, _ = oracle.attn_row(cache2, q.to(torch.bfloat16), table, torch.tensor([L], dtype=torch.int32),
                                  torch.tensor([0, 1], dtype=torch.int32), 1, 1000.0, 0, 0, 0)
    np.testing.assert_allclose(out, vals[pos, 0].double().numpy(), rtol=0, atol=1e-12)


def test_block_count_from_the_pages():
    g = golden("block_count.json")
    B, n = g["block_size"], g["new_tokens"]
    assert math.ceil(n / B) == g["blocks"]
    # a 17-token request reads exactly two table entries: entry 2 may hold
    # garbage (-1) and only slot 0 of the second block is read
    step = custom([(n - 1, 1)], 2, 2, 64, seed=3)
    assert int((step.block_tables[0] >= 0).sum()) == g["blocks"]
    cache, out, _ = oracle.run_step(step)
    assert np.isfinite(out).all()
    second = int(step.block_tables[0, 1])
    written = np.argwhere(cache[second] != 0x7FC0)
    assert set(written[:, 2].tolist()) == {0}


def test_kv_bytes_formula_from_the_pages():
    g = golden("kv_bytes.json")
    m = g["llama13b"]
    per_token = 2 * m["num_layers"] * m["num_kv_heads"] * m["head_size"] * g["dtype_bytes"]
    assert per_token == g["kv_bytes_per_token_13b"]
    assert abs(per_token - g["kv_bytes_per_token_13b_stated_approx"]) / per_token < 0.03
    assert abs(per_token * 2048 - g["tokens_2048_bytes_stated_approx"]) / (per_token * 2048) < 0.05
    # the cache layout uses exactly the formula's bytes per block
    B = g["block_size"]
    per_block = 2 * B * m["num_kv_heads"] * m["head_size"] * g["dtype_bytes"]
    cache = oracle.new_cache(3, m["num_kv_heads"], m["head_size"], B)
    assert cache.nbytes == 3 * per_block
    step = wl.make_workload("tiny-decode")
    assert step.pool_bytes() == step.num_blocks * 2 * B * step.num_kv_heads * step.head_size * 2


def test_cow_fork_construction_matches_the_pages():
    g = golden("cow_example.json")
    # our generator's fork: the parent's table except its last block, which is
    # a fresh block holding a copy of the parent's last block's cached tokens
    reqs = [wl.RequestSpec(3 * 16 - 1, 1)]      # a 3-block request
    step = wl.build_step("cow", reqs, 2, 2, 64, 16, 5, forks=[0, 0, 0], permute_blocks=False)
    tables = step.block_tables.tolist()
    assert tables[0] == g["prompt_blocks"]
    refs = {b: 0 for b in range(16)}
    for t in tables:
        for b in t:
            refs[b] += 1
    n = g["n_samples"]
    assert [refs[b] for b in g["prompt_blocks"][:2]] == g["ref_counts_after_fork"][:2]
    assert refs[g["prompt_blocks"][2]] == g["ref_counts_after_sample0_write"][2] - (n - 1) + 1
    for t in tables[1:]:
        assert t[:2] == g["prompt_blocks"][:2] and t[2] not in g["prompt_blocks"]
    # copies hold the same cached tokens, so every fork sees the parent's keys
    cache, out, _ = oracle.run_step(step)
    for f in range(1, 4):
        src, dst = tables[0][2], tables[f][2]
        assert (cache[dst][:, :, :15] == cache[src][:, :, :15]).all()


def test_chunk_budget_shapes_the_mixed_step():
    g = golden("chunk_budget.json")
    ex = g["tutorial_example"]
    assert g["token_budget"] - ex["num_decodes"] == ex["chunk"]
    ms = g["mixed_step"]
    first = min(ms["prompt_len"], g["token_budget"] - ms["num_decodes"])
    assert first == ms["first_chunk"] and ms["prompt_len"] - first == ms["second_chunk"]
    step = wl.make_workload("llama3-8b-mixed")
    ql = step.query_lens.tolist()
    assert ql == [1, 1, ms["first_chunk"]] and step.num_tokens == g["token_budget"]
    assert step.context_lens.tolist() == [699, 1499, 0]


# ---------------------------------------------------------------------------
# closed forms and invariants
# ---------------------------------------------------------------------------

def test_single_key_returns_its_value_exactly():
    step = custom([(0, 1), (0, 1)], 4, 2, 128, seed=11)
    _, out, lse = oracle.run_step(step)
    G = 2
    for r in range(2):
        k, v = step.request_kv(r)
        for h in range(4):
            assert (out[r, h] == v[0, h // G].double().numpy()).all()
            s = step.scale * float((step.query[r, h].double() * k[0, h // G].double()).sum())
            assert abs(lse[r, h] - s) <= 1e-12 * max(1.0, abs(s))


def test_two_keys_closed_form():
    step = custom([(1, 1)], 2, 1, 64, seed=12)
    _, out, _ = oracle.run_step(step)
    k, v = step.request_kv(0)
    for h in range(2):
        q = step.query[0, h].double()
        s0 = step.scale * float((q * k[0, 0].double()).sum())
        s1 = step.scale * float((q * k[1, 0].double()).sum())
        sig = 1.0 / (1.0 + math.exp(s1 - s0))
        expect = sig * v[0, 0].double().numpy() + (1.0 - sig) * v[1, 0].double().numpy()
        np.testing.assert_allclose(out[0, h], expect, rtol=1e-12, atol=1e-13)


def test_uniform_keys_and_zero_scale_give_the_mean_of_values():
    step = custom([(37, 1), (5, 9)], 4, 2, 64, seed=13)
    cache = oracle.new_cache(step.num_blocks, step.num_kv_heads, step.head_size)
    # every key equal: overwrite all keys with the same vector
    same = step.hist_key[:1].expand(step.hist_key.shape[0], -1, -1).contiguous()
    same_new = step.hist_key[:1].expand(step.key.shape[0], -1, -1).contiguous()
    oracle.kv_write(cache, same, step.hist_value, step.hist_slot_mapping)
    oracle.kv_write(cache, same_new, step.value, step.slot_mapping)
    out, _ = oracle.paged_attn(cache, step.query, step.block_tables, step.seq_lens,
                               step.query_start_loc, step.num_q_heads, step.scale)
    _, out0, _ = (None, *oracle.paged_attn(oracle.run_step(step)[0], step.query, step.block_tables,
                                           step.seq_lens, step.query_start_loc, step.num_q_heads, 0.0))
    for r in range(step.num_seqs):
        _, v = step.request_kv(r)
        q0, q1 = int(step.query_start_loc[r]), int(step.query_start_loc[r + 1])
        c = int(step.seq_lens[r]) - (q1 - q0)
        for i in range(q1 - q0):
            for h in range(4):
                mean = v[:c + i + 1, h // 2].double().mean(0).numpy()
                np.testing.assert_allclose(out[q0 + i, h], mean, rtol=1e-12, atol=1e-13)
                np.testing.assert_allclose(out0[q0 + i, h], mean, rtol=1e-12, atol=1e-13)


def test_weights_sum_to_one_and_are_nonnegative():
    step = custom([(70, 3)], 4, 4, 64, seed=14)
    cache, _, _ = oracle.run_step(step)
    for i in range(3):
        for h in range(4):
            _, _, w = oracle.attn_row(cache, step.query, step.block_tables, step.seq_lens,
                                      step.query_start_loc, 4, step.scale, 0, i, h, want_weights=True)
            assert w.shape[0] == 70 + i + 1
            assert (w >= 0).all()
            assert abs(w.sum() - 1.0) <= 1e-12


def test_output_is_unchanged_by_relabelling_physical_blocks():
    step = custom([(50, 1), (3, 20), (31, 2)], 8, 2, 64, seed=15)
    cache, out, lse = oracle.run_step(step)
    perm = np.random.default_rng(5).permutation(step.num_blocks)
    cache2 = np.empty_like(cache)
    cache2[perm] = cache
    bt = step.block_tables.numpy()
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    out2, lse2 = oracle.paged_attn(cache2, step.query, bt2, step.seq_lens, step.query_start_loc,
                                   step.num_q_heads, step.scale)
    assert (out2 == out).all() and (lse2 == lse).all()


def test_shared_prefix_equals_private_copies():
    reqs = [(40, 1), (65, 2), (33, 1)]
    shared = custom(reqs, 4, 2, 64, seed=16, shared_prefix_len=32)
    cache, out, _ = oracle.run_step(shared)
    # private copies: give every request its own copy of the prefix blocks
    nb = shared.num_blocks
    extra = 2 * shared.num_seqs
    cache2 = np.concatenate([cache, oracle.new_cache(extra, 2, 64)], axis=0)
    bt2 = shared.block_tables.numpy().copy()
    nxt = nb
    for r in range(shared.num_seqs):
        for b in range(2):
            cache2[nxt] = cache[bt2[r, b]]
            bt2[r, b] = nxt
            nxt += 1
    assert len(set(bt2[:, :2].flatten().tolist())) == 2 * shared.num_seqs
    out2, _ = oracle.paged_attn(cache2, shared.query, bt2, shared.seq_lens, shared.query_start_loc,
                                4, shared.scale)
    assert (out2 == out).all()


def test_split_key_range_merges_to_the_full_row():
    step = custom([(150, 2)], 4, 1, 128, seed=17)
    cache, out, lse = oracle.run_step(step)
    rng = np.random.default_rng(9)
    for i in range(2):
        L = 150 + i + 1
        for h in range(4):
            cuts = sorted(set(rng.integers(1, L, size=4).tolist()))
            bounds = [0] + cuts + [L + 5]          # the last part runs past the row's keys
            parts_o, parts_l = [], []
            for a, b in zip(bounds[:-1], bounds[1:]):
                o, l, _ = oracle.attn_row(cache, step.query, step.block_tables, step.seq_lens,
                                          step.query_start_loc, 4, step.scale, 0, i, h, a, b)
                parts_o.append(o)
                parts_l.append(l)
            # an empty part (no visible key) carries lse = -inf and weight 0
            o, l, _ = oracle.attn_row(cache, step.query, step.block_tables, step.seq_lens,
                                      step.query_start_loc, 4, step.scale, 0, i, h, L + 10, L + 20)
            assert l == -math.inf and (o == 0).all()
            parts_o.append(o)
            parts_l.append(l)
            mo, ml = oracle.lse_combine(np.stack(parts_o), np.array(parts_l))
            np.testing.assert_allclose(mo, out[i, h], rtol=1e-12, atol=1e-13)
            assert abs(ml - lse[i, h]) <= 1e-12 * abs(lse[i, h]) + 1e-12


def test_kv_write_round_trip_and_untouched_slots():
    step = custom([(10, 5), (0, 3)], 2, 2, 64, seed=18)
    cache = oracle.new_cache(step.num_blocks, 2, 64)
    before = cache.copy()
    slots = step.slot_mapping.clone()
    slots[1] = -1                                    # a padding token is skipped
    oracle.kv_write(cache, step.key, step.value, slots)
    raw_k = step.key.view(torch.int16).numpy().view(np.uint16)
    raw_v = step.value.view(torch.int16).numpy().view(np.uint16)
    touched = np.zeros(cache.shape[:1] + cache.shape[3:4], dtype=bool)  # [block, offset]
    for t, s in enumerate(slots.tolist()):
        if s < 0:
            continue
        b, o = divmod(s, 16)
        assert (cache[b, :, 0, o] == raw_k[t]).all() and (cache[b, :, 1, o] == raw_v[t]).all()
        touched[b, o] = True
    mask = ~touched[:, None, None, :, None].repeat(2, 1).repeat(2, 2).repeat(64, 4)
    assert (cache[mask] == before[mask]).all()
    b1, o1 = divmod(int(step.slot_mapping[1]), 16)
    assert (cache[b1, :, :, o1] == 0x7FC0).all()


def test_kv_write_rejects_duplicates_and_out_of_range():
    cache = oracle.new_cache(4, 1, 64)
    k = torch.zeros(2, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(oracle.OracleError):
        oracle.kv_write(cache, k, k, torch.tensor([5, 5]))
    with pytest.raises(oracle.OracleError):
        oracle.kv_write(cache, k, k, torch.tensor([5, 64]))
    oracle.kv_write(cache, k, k, torch.tensor([-1, -1]))
    assert (cache == 0x7FC0).all()


def test_nan_slots_never_reach_the_output():
    # a partial last block: slots past seq_len stay NaN in the oracle's cache
    step = custom([(16, 1), (3, 30)], 4, 1, 64, seed=19)
    cache, out, _ = oracle.run_step(step)
    nan_blocks = (cache == 0x7FC0).any(axis=(1, 2, 4))
    assert nan_blocks.any()
    assert np.isfinite(out).all()


def test_wrong_metadata_is_rejected():
    step = custom([(5, 2)], 2, 1, 64, seed=20)
    cache, _, _ = oracle.run_step(step)
    bad_sl = step.seq_lens.clone()
    bad_sl[0] = 1                                    # seq_len < query_len
    with pytest.raises(oracle.OracleError):
        oracle.paged_attn(cache, step.query, step.block_tables, bad_sl, step.query_start_loc, 2, 1.0)
    bad_bt = step.block_tables.clone()
    bad_bt[0, 0] = step.num_blocks                   # out of the pool
    with pytest.raises(oracle.OracleError):
        oracle.paged_attn(cache, step.query, bad_bt, step.seq_lens, step.query_start_loc, 2, 1.0)
    cache2 = oracle.new_cache(step.num_blocks, 2, 64)
    with pytest.raises(oracle.OracleError):          # q heads not a multiple of kv heads
        oracle.paged_attn(cache2, torch.zeros(2, 3, 64, dtype=torch.bfloat16), step.block_tables,
                          step.seq_lens, step.query_start_loc, 3, 1.0)


def test_copy_on_write_copy_gives_the_fork_the_parents_view():
    """The COW walk-through of the pages: block 2 copied into block 7; the fork's
    table [0, 1, 7] then reads exactly what the parent's [0, 1, 2] reads."""
    g = golden("cow_example.json")
    d, hkv, H = 64, 2, 4
    step = wl.build_step("cow2", [wl.RequestSpec(3 * 16 - 2, 1)], H, hkv, d, 16, 31, permute_blocks=False)
    assert step.block_tables[0].tolist() == g["prompt_blocks"]
    cache, out, _ = oracle.run_step(step)
    oracle.copy_blocks(cache, torch.tensor([[g["prompt_blocks"][2], g["sample0_new_block"]]]))
    assert (cache[g["sample0_new_block"]] == cache[g["prompt_blocks"][2]]).all()
    fork_table = torch.tensor([g["sample0_table_after_write"]], dtype=torch.int32)
    out2, _ = oracle.paged_attn(cache, step.query, fork_table, step.seq_lens, step.query_start_loc, H, step.scale)
    assert (out2 == out).all()
    # other blocks untouched, out-of-range pairs refused
    before = cache.copy()
    with pytest.raises(oracle.OracleError):
        oracle.copy_blocks(cache, torch.tensor([[0, 16]]))
    assert (cache == before).all()

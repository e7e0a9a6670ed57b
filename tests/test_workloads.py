"""The seeded input generator: shapes, determinism, structure of the named workloads."""

import math

import torch

import workloads as wl


def test_same_seed_same_inputs():
    a = wl.make_workload("tiny-decode")
    b = wl.make_workload("tiny-decode")
    for f in ("seq_lens", "query_start_loc", "block_tables", "slot_mapping", "hist_slot_mapping"):
        assert torch.equal(getattr(a, f), getattr(b, f))
    for f in ("query", "key", "value", "hist_key", "hist_value"):
        assert torch.equal(getattr(a, f).view(torch.int16), getattr(b, f).view(torch.int16))


def test_slots_are_unique_and_inside_the_tables():
    for name in ("tiny-decode", "tinyllama-decode", "llama3-8b-mixed", "llama3-70b-prefix"):
        s = wl.make_workload(name)
        B = s.block_size
        all_slots = torch.cat([s.hist_slot_mapping, s.slot_mapping])
        assert torch.unique(all_slots).numel() == all_slots.numel()
        assert int(all_slots.min()) >= 0 and int(all_slots.max()) < s.num_blocks * B
        # every new token's slot is its position's slot in its own table
        for r in range(s.num_seqs):
            q0, q1 = int(s.query_start_loc[r]), int(s.query_start_loc[r + 1])
            c = int(s.seq_lens[r]) - (q1 - q0)
            for i in range(q1 - q0):
                pos = c + i
                assert int(s.slot_mapping[q0 + i]) == int(s.block_tables[r, pos // B]) * B + pos % B
        # tables list exactly ceil(seq_len / 16) blocks, the rest is -1
        for r in range(s.num_seqs):
            nb = math.ceil(int(s.seq_lens[r]) / B)
            assert bool((s.block_tables[r, :nb] >= 0).all()) and bool((s.block_tables[r, nb:] == -1).all())


def test_named_workload_shapes():
    s = wl.make_workload("tiny-decode")
    assert (s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_size, s.num_blocks) == (4, 8, 8, 64, 64)
    assert int(s.seq_lens.min()) >= 1 and int(s.seq_lens.max()) <= 128
    s = wl.make_workload("tinyllama-decode")
    assert (s.num_seqs, s.num_q_heads, s.num_kv_heads, s.head_size, s.num_blocks) == (64, 32, 4, 64, 16384)
    assert int(s.seq_lens.min()) >= 512 and int(s.seq_lens.max()) <= 2048
    s = wl.make_workload("llama3-8b-mixed")
    assert s.query_start_loc.tolist() == [0, 1, 2, 2048] and s.seq_lens.tolist() == [700, 1500, 2046]
    s = wl.make_workload("llama3-70b-prefix")
    assert s.num_seqs == 72 and (s.num_q_heads, s.num_kv_heads) == (64, 8)
    prefix = s.block_tables[:, :64]
    assert bool((prefix == prefix[0]).all())                   # one shared 1024-token prefix
    for f in range(8):                                         # forks: all but the last block
        nb = math.ceil(int(s.seq_lens[f]) / 16)
        assert torch.equal(s.block_tables[64 + f, :nb - 1], s.block_tables[f, :nb - 1])
        assert int(s.block_tables[64 + f, nb - 1]) != int(s.block_tables[f, nb - 1])
        assert int(s.seq_lens[64 + f]) == int(s.seq_lens[f])


def test_lognormal_lengths_of_the_13b_batch():
    # draws only the lengths (same generator order as the full workload)
    gen = torch.Generator().manual_seed(wl.seed_of("llama13b-decode"))
    sigma = 0.8
    mu = math.log(800.0) - sigma * sigma / 2
    z = torch.randn(256, generator=gen, dtype=torch.float64)
    L = torch.clamp(torch.round(torch.exp(mu + sigma * z)), 16, 4096)
    assert 600 < float(L.mean()) < 1000
    assert int(L.min()) >= 16 and int(L.max()) <= 4096


def test_subset_keeps_each_requests_values():
    s = wl.make_workload("llama3-70b-prefix")
    sub = s.subset([3, 64, 70])
    assert sub.num_seqs == 3
    for new_r, old_r in enumerate([3, 64, 70]):
        k0, v0 = s.request_kv(old_r)
        k1, v1 = sub.request_kv(new_r)
        assert torch.equal(k0.view(torch.int16), k1.view(torch.int16))
        assert torch.equal(v0.view(torch.int16), v1.view(torch.int16))
    assert sub.num_blocks < s.num_blocks

"""kv_write on the GPU against the oracle's cache write: bit-exact."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import new_pool, to_dev, write_history

pytestmark = pytest.mark.gpu


def raw(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("name", ["tiny-decode", "tinyllama-decode", "llama3-8b-mixed"])
def test_whole_pool_bit_exact(name):
    step = wl.make_workload(name)
    dev = to_dev(step)
    pool = new_pool(step)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    torch.cuda.synchronize()
    ref = oracle.new_cache(step.num_blocks, step.num_kv_heads, step.head_size)
    oracle.kv_write(ref, step.hist_key, step.hist_value, step.hist_slot_mapping)
    oracle.kv_write(ref, step.key, step.value, step.slot_mapping)
    assert np.array_equal(raw(pool), ref)


@pytest.mark.parametrize("name", ["llama3-70b-prefix", "llama13b-decode"])
def test_full_size_every_used_block_bit_exact(name):
    """Full-size pools (13-33 GB): every block any table uses, against the
    oracle's write of the whole step into a pool compacted to those blocks,
    and a sample of never-used blocks (still the NaN poison)."""
    step = wl.make_workload(name)
    dev = to_dev(step)
    pool = new_pool(step)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    torch.cuda.synchronize()
    del dev
    S = step.num_seqs
    sub = step.subset(range(S))
    ref = oracle.new_cache(sub.num_blocks, sub.num_kv_heads, sub.head_size)
    oracle.kv_write(ref, sub.hist_key, sub.hist_value, sub.hist_slot_mapping)
    oracle.kv_write(ref, sub.key, sub.value, sub.slot_mapping)
    # the subset renumbers blocks in order of first appearance in the tables
    order = []
    seen = set()
    for r in range(S):
        nb = (int(step.seq_lens[r]) + 15) // 16
        for b in step.block_tables[r, :nb].tolist():
            if b not in seen:
                seen.add(b)
                order.append(b)
    assert len(order) == sub.num_blocks
    idx = torch.tensor(order, device=pool.device)
    for a in range(0, len(order), 4096):          # a few hundred MB of the pool at a time
        got = raw(pool[idx[a:a + 4096]])
        assert np.array_equal(got, ref[a:a + 4096]), f"blocks {a}..{a + 4095} of the used set differ"
    used = torch.zeros(step.num_blocks, dtype=torch.bool)
    used[torch.tensor(order)] = True
    free = torch.nonzero(~used).flatten()
    pick = free[torch.randperm(free.numel(), generator=torch.Generator().manual_seed(1))[:64]]
    assert (raw(pool[pick.to(pool.device)]) == 0x7FC0).all()


def test_padding_and_strided_views_and_bad_slots():
    step = wl.build_step("pad", [wl.RequestSpec(5, 7), wl.RequestSpec(0, 9)], 4, 2, 128, 16, 3)
    T = step.num_tokens
    # K and V as views of a fused [T, (H + 2 Hkv) d] buffer
    qkv = torch.randn(T, (4 + 4) * 128, dtype=torch.float32).to(torch.bfloat16)
    qkv[:, 4 * 128:6 * 128] = step.key.reshape(T, -1)
    qkv[:, 6 * 128:] = step.value.reshape(T, -1)
    qkv = qkv.cuda()
    k = qkv[:, 4 * 128:6 * 128].view(T, 2, 128)
    v = qkv[:, 6 * 128:].view(T, 2, 128)
    slots = step.slot_mapping.clone()
    slots[3] = -1
    slots[5] = step.num_blocks * 16 + 7          # outside the pool: skipped, reported
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pool = new_pool(step)
    pkv.kv_write(pool, k, v, slots.cuda(), device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 7                # PKV_ERR_DEVICE_INDEX
    ref = oracle.new_cache(step.num_blocks, 2, 128)
    ok = slots.clone()
    ok[5] = -1
    oracle.kv_write(ref, step.key, step.value, ok)
    assert np.array_equal(raw(pool), ref)


def test_host_side_errors_enqueue_nothing():
    pool = torch.zeros(4, 2, 2, 16, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(3, 2, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(3, dtype=torch.int64, device="cuda")
    lib = pkv.load()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.pkv_kv_write(pool.data_ptr(), 4, 2, 96, 16, k.data_ptr(), 256, k.data_ptr(), 256,
                            s.data_ptr(), 3, None, stream) == 3
    assert lib.pkv_kv_write(pool.data_ptr(), 4, 2, 128, 8, k.data_ptr(), 256, k.data_ptr(), 256,
                            s.data_ptr(), 3, None, stream) == 3
    assert lib.pkv_kv_write(pool.data_ptr() + 2, 4, 2, 128, 16, k.data_ptr(), 256, k.data_ptr(), 256,
                            s.data_ptr(), 3, None, stream) == 4
    assert lib.pkv_kv_write(pool.data_ptr(), 4, 2, 128, 16, k.data_ptr(), 100, k.data_ptr(), 256,
                            s.data_ptr(), 3, None, stream) == 2
    assert (pool == 0).all()

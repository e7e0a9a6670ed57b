"""Copy-on-write block copies on the GPU against the oracle's copy: bit-exact."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import new_pool, to_dev, write_history

pytestmark = pytest.mark.gpu


def raw(t):
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("d,hkv", [(64, 4), (128, 8)])
def test_copy_blocks_bit_exact(d, hkv):
    step = wl.build_step("cp", [wl.RequestSpec(100, 1), wl.RequestSpec(37, 2), wl.RequestSpec(64, 1)],
                         2 * hkv, hkv, d, 64, 17)
    dev = to_dev(step)
    pool = new_pool(step)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    ref = oracle.new_cache(step.num_blocks, hkv, d)
    oracle.kv_write(ref, step.hist_key, step.hist_value, step.hist_slot_mapping)
    oracle.kv_write(ref, step.key, step.value, step.slot_mapping)
    used = sorted(set(step.block_tables[step.block_tables >= 0].tolist()))
    free = [b for b in range(step.num_blocks) if b not in used]
    rng = np.random.default_rng(4)
    src = rng.choice(used, size=6, replace=False)
    dst = rng.choice(free, size=6, replace=False)
    mapping = torch.tensor(np.stack([src, dst], axis=1), dtype=torch.int64)
    pkv.copy_blocks(pool, mapping.cuda())
    oracle.copy_blocks(ref, mapping)
    torch.cuda.synchronize()
    assert np.array_equal(raw(pool), ref)


def test_copy_blocks_fork_then_attend_matches_oracle():
    # a parent and a fork sharing all but the last block: the fork's last block
    # is made on the GPU by copy_blocks, then both write their own new token
    from tolerance import check_close
    parent = wl.build_step("par", [wl.RequestSpec(75, 1)], 8, 2, 128, 32, 23, forks=[0], permute_blocks=False)
    tables = parent.block_tables
    fork_last = int(tables[1, -1])
    parent_last = int(tables[0, -1])
    dev = to_dev(parent)
    pool = new_pool(parent)
    # history without the fork's copied entries: the copy is done by copy_blocks
    keep = torch.div(parent.hist_slot_mapping, 16, rounding_mode="floor") != fork_last
    pkv.kv_write(pool, dev["hist_key"][keep.cuda()].contiguous(), dev["hist_value"][keep.cuda()].contiguous(),
                 dev["hist_slot_mapping"][keep.cuda()].contiguous())
    pkv.copy_blocks(pool, torch.tensor([[parent_last, fork_last]], dtype=torch.int64, device="cuda"))
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    n = pkv.paged_attn_workspace_size(2, 2, 1, parent.max_seq_len, 8, 2, 128)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.empty(2, 8, 128, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn(out, dev["query"], pool, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                   1, parent.max_seq_len, parent.scale, ws)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    _, ref, _ = oracle.run_step(parent)
    check_close(out, ref, "fork after copy")


def test_copy_blocks_bad_ids_are_skipped_and_reported():
    pool = torch.zeros(8, 2, 2, 16, 64, dtype=torch.bfloat16, device="cuda")
    pool[3].fill_(1.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.copy_blocks(pool, torch.tensor([[3, 5], [3, 8], [-1, 2]], dtype=torch.int64, device="cuda"), status)
    torch.cuda.synchronize()
    assert int(status.item()) == 7
    assert (pool[5] == 1.0).all() and (pool[2] == 0).all()

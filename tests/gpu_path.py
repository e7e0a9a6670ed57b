"""Runs a ``workloads.Step`` through the CUDA library (tests' helper).

The pool starts as bf16 NaN on the device; history entries and then the
step's new tokens are written with the library's own kv_write, then
paged_attn and paged_attn_combine run on the current stream.
"""

import torch

import paged_kv_cache_111_gb300 as pkv
import workloads as wl


def to_dev(step: wl.Step, device="cuda"):
    d = {}
    for f in ("seq_lens", "query_start_loc", "block_tables", "query", "key", "value", "slot_mapping",
              "hist_key", "hist_value", "hist_slot_mapping"):
        d[f] = getattr(step, f).to(device).contiguous()
    return d


def new_pool(step: wl.Step, device="cuda") -> torch.Tensor:
    return wl.make_poisoned_pool_like(step, device=device)


def write_history(step: wl.Step, pool: torch.Tensor, dev: dict, chunk_tokens: int = 1 << 16) -> None:
    C = dev["hist_slot_mapping"].shape[0]
    for a in range(0, C, chunk_tokens):
        b = min(C, a + chunk_tokens)
        pkv.kv_write(pool, dev["hist_key"][a:b], dev["hist_value"][a:b], dev["hist_slot_mapping"][a:b])


def workspace_for(step: wl.Step, device="cuda") -> torch.Tensor:
    n = pkv.paged_attn_workspace_size(step.num_seqs, step.num_tokens, step.max_query_len, step.max_seq_len,
                                      step.num_q_heads, step.num_kv_heads, step.head_size)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def attend(step: wl.Step, pool: torch.Tensor, dev: dict, ws: torch.Tensor, num_splits: int = 0,
           out: torch.Tensor = None) -> torch.Tensor:
    if out is None:
        out = torch.full((step.num_tokens, step.num_q_heads, step.head_size), float("nan"),
                         dtype=torch.bfloat16, device=pool.device)
    pkv.paged_attn(out, dev["query"], pool, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                   step.max_query_len, step.max_seq_len, step.scale, ws, num_splits=num_splits)
    pkv.paged_attn_combine(out, ws)
    return out


def run_step(step: wl.Step, num_splits: int = 0, device="cuda"):
    """Returns (pool, out, workspace status) with pool and out still on the device."""
    dev = to_dev(step, device)
    pool = new_pool(step, device)
    write_history(step, pool, dev)
    pkv.kv_write(pool, dev["key"], dev["value"], dev["slot_mapping"])
    ws = workspace_for(step, device)
    out = attend(step, pool, dev, ws, num_splits)
    torch.cuda.synchronize()
    return pool, out, pkv.workspace_status(ws)

"""A layer-step (kv_write + paged_attn + paged_attn_combine) captured in a CUDA
graph and replayed on new inputs of the same shapes matches the oracle.

Decode steps are captured once per batch size and replayed every step
("Inside vLLM: Anatomy of a High-Throughput LLM Inference System", the
captured execution mode; "vLLM source reading", section 5.2).  The step's
calls are capturable: the plan is computed on the GPU from the device
metadata, so new lengths, tables and slots take effect on replay.  The same
holds over an E4M3 cache with fixed per-tensor scales.
"""

import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import new_pool, to_dev, write_history
from tolerance import check_close

pytestmark = pytest.mark.gpu


def make(seed, extra=0):
    # decode rows, a multi-token (speculative-verify) row and a short chunk
    reqs = [wl.RequestSpec(300 + extra, 1), wl.RequestSpec(47, 4), wl.RequestSpec(16, 1), wl.RequestSpec(5, 9)]
    return wl.build_step("graph", reqs, 16, 2, 128, 256, seed, extra_table_cols=16)


def test_captured_step_replays_on_new_inputs():
    base = make(1)
    dev = to_dev(base)
    static = {k: v.clone() for k, v in dev.items()}
    pool = new_pool(base)
    maxq = 16
    maxs = static["block_tables"].shape[1] * 16          # what the captured table can hold
    n = pkv.paged_attn_workspace_size(base.num_seqs, base.num_tokens, maxq, maxs, 16, 2, 128)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.empty(base.num_tokens, 16, 128, dtype=torch.bfloat16, device="cuda")

    def layer_step():
        pkv.kv_write(pool, static["key"], static["value"], static["slot_mapping"])
        pkv.paged_attn(out, static["query"], pool, static["block_tables"], static["seq_lens"],
                       static["query_start_loc"], maxq, maxs, base.scale, ws)
        pkv.paged_attn_combine(out, ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer_step()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer_step()

    for seed, extra in ((2, 0), (3, 17), (4, 100)):
        step = make(seed, extra)
        assert step.num_tokens == base.num_tokens and step.max_seq_len <= maxs
        d = to_dev(step)
        pool.view(torch.int16).fill_(wl.BF16_NAN_BITS)
        write_history(step, pool, d)                   # this step's cached tokens
        for k in ("key", "value", "slot_mapping", "query", "seq_lens", "query_start_loc"):
            static[k].copy_(d[k])
        static["block_tables"].fill_(-1)
        cols = min(static["block_tables"].shape[1], d["block_tables"].shape[1])
        static["block_tables"][:, :cols].copy_(d["block_tables"][:, :cols])
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert pkv.workspace_status(ws) == 0
        _, ref, _ = oracle.run_step(step)
        check_close(out, ref, f"replay seed {seed}")


def test_captured_step_replays_on_new_inputs_fp8():
    base = make(11)
    dev = to_dev(base)
    static = {k: v.clone() for k, v in dev.items()}
    cache = torch.full(base.pool_shape(), 0x7F, dtype=torch.uint8, device="cuda")
    ks, vs = 0.013, 0.017
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    maxq = 16
    maxs = static["block_tables"].shape[1] * 16
    n = pkv.paged_attn_workspace_size(base.num_seqs, base.num_tokens, maxq, maxs, 16, 2, 128)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.empty(base.num_tokens, 16, 128, dtype=torch.bfloat16, device="cuda")

    def layer_step():
        pkv.kv_write_fp8(cache, static["key"], static["value"], static["slot_mapping"], ks, vs, st)
        pkv.paged_attn_fp8(out, static["query"], cache, static["block_tables"], static["seq_lens"],
                           static["query_start_loc"], maxq, maxs, base.scale, ks, vs, ws)
        pkv.paged_attn_combine(out, ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer_step()                                   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer_step()

    for seed, extra in ((12, 0), (13, 41)):
        step = make(seed, extra)
        assert step.num_tokens == base.num_tokens and step.max_seq_len <= maxs
        d = to_dev(step)
        cache.fill_(0x7F)
        C = d["hist_slot_mapping"].shape[0]
        if C:
            pkv.kv_write_fp8(cache, d["hist_key"], d["hist_value"], d["hist_slot_mapping"], ks, vs, st)
        for k in ("key", "value", "slot_mapping", "query", "seq_lens", "query_start_loc"):
            static[k].copy_(d[k])
        static["block_tables"].fill_(-1)
        cols = min(static["block_tables"].shape[1], d["block_tables"].shape[1])
        static["block_tables"][:, :cols].copy_(d["block_tables"][:, :cols])
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert int(st.item()) == 0 and pkv.workspace_status(ws) == 0
        _, ref, _ = oracle.run_step_fp8(step, ks, vs)
        check_close(out, ref, f"fp8 replay seed {seed}")


"""Benchmark of one paged-attention layer-step on GB300.

A step is one pass of the whole hot path over one batch: the cache write of
the step's new tokens (kv_write), paged attention (paged_attn) and the
split merge (paged_attn_combine), on inputs already resident in HBM.

Default workload: the LLaMA-13B-shaped decode batch (256 requests, 40 q = 40
kv heads, head size 128, lognormal lengths around 800 tokens, 100000-block
cache, about 4.1 GB of KV read per step).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle on host cores

For N > 1 (torchrun, one rank per GPU) every rank runs its own replica of
the batch (independent requests, weak scaling); no collective touches the
data path, only the barrier and the max of the ranks' times.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "decode paged-attn achieved HBM GB/s (% of peak), tokens/s per layer-step"
FALLBACK_HBM_GBS = 6800.0
SETTLE_S = 1.5          # seconds of untimed steps under the clock sampler before the timed passes

# DRAM bytes (read + write) per algorithmic byte of the attention call, from
# ncu captures (dram__bytes_read.sum + dram__bytes_write.sum of the kernels
# of one call, over the call's algorithmic bytes) of smaller cases of the same
# kernels.  Traffic grows with the KV bytes read, so a full launch's traffic is
# the ratio times its algorithmic bytes.  A ratio holds only for the kernel
# sources it was measured on (hash of the files below); otherwise null.
TRAFFIC_SOURCES = ("decode.cu", "pkv_common.cuh", "paged_attn.cu", "prefill_tc.cu", "prefill_sk.cu",
                   "prefill_common.cuh", "tc_common.cuh", "attn_internal.cuh")
TRAFFIC = {
    # "<cache> <kernels of the call>": decode (plan + decode), cascade (plus the
    # shared-prefix pass), prefill (plus the tcgen05 chunk kernel).  ratio =
    # (dram__bytes_read.sum + dram__bytes_write.sum of the call's kernels, one
    # call, ncu with its default cache flush) / the call's algorithmic bytes.
    # Writes that stay in L2 until after the kernel do not count, so a call
    # whose output is large (a prefill chunk) reads below 1.
    "bf16 decode": {"sources_sha256_16": "f1eb5d212e731fb2", "ratio": 1045.1558e6 / 1033884588,
                    "source": "ncu DRAM counters of plan + decode on llama13b-decode, first 64 requests"},
    "e4m3 decode": {"sources_sha256_16": "f1eb5d212e731fb2", "ratio": 524.2228e6 / 517604268,
                    "source": "ncu DRAM counters of plan + decode on llama13b-decode, first 64 requests, E4M3"},
    "bf16 cascade": {"sources_sha256_16": "f1eb5d212e731fb2", "ratio": 29.5035e6 / 28294800,
                     "source": "ncu DRAM counters of plan + decode + shared-prefix pass on llama3-70b-prefix, "
                               "first 24 requests"},
    "e4m3 cascade": {"sources_sha256_16": "f1eb5d212e731fb2", "ratio": 15.2649e6 / 14544528,
                     "source": "ncu DRAM counters of plan + decode + shared-prefix pass on llama3-70b-prefix, "
                               "first 24 requests, E4M3"},
    "bf16 prefill": {"sources_sha256_16": "f1eb5d212e731fb2", "ratio": 34.3981e6 / 50947140,
                     "source": "ncu DRAM counters of plan + decode + prefill on llama3-8b-mixed"},
    "e4m3 prefill": {"sources_sha256_16": "f1eb5d212e731fb2", "ratio": 25.7139e6 / 42251332,
                     "source": "ncu DRAM counters of plan + decode + prefill on llama3-8b-mixed, E4M3"},
}


def percentiles(values, fractions=(0.1, 0.5, 0.9)):
    """Nearest-rank percentiles of a non-empty list (each fraction in [0, 1])."""
    q = sorted(values)
    return [q[min(len(q) - 1, max(0, math.ceil(f * len(q)) - 1))] for f in fractions]


def attention_sources_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in TRAFFIC_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_111_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def algorithmic_bytes(step: wl.Step, kv_elem_bytes: int = 2) -> dict:
    """Bytes the method must move per step (each byte once), by phase.

    attention: K and V of every key each request sees (a physical block
    shared by several requests counts once), Q in, out, the table entries
    read and the per-request lengths.  kv_write: new K/V read (bf16) and
    written (kv_elem_bytes per element: 2 for bf16, 1 for E4M3), and slot
    numbers.
    """
    H, Hkv, d, B = step.num_q_heads, step.num_kv_heads, step.head_size, step.block_size
    T, S = step.num_tokens, step.num_seqs
    per_token_kv = 2 * Hkv * d * kv_elem_bytes
    # unique (block, used tokens): a shared block is read once
    used = {}
    for r in range(S):
        L = int(step.seq_lens[r])
        nb = (L + B - 1) // B
        for i, b in enumerate(step.block_tables[r, :nb].tolist()):
            n = min(B, L - i * B)
            used[b] = max(used.get(b, 0), n)
    kv_unique = sum(used.values()) * per_token_kv
    kv_logical = int(step.seq_lens.long().sum()) * per_token_kv
    tables = sum((int(l) + B - 1) // B for l in step.seq_lens.tolist()) * 4
    attn = kv_unique + 2 * T * H * d * 2 + tables + 4 * S + 4 * (S + 1)
    kvw = T * 2 * Hkv * d * 2 + T * per_token_kv + 8 * T
    # flops: every query row of every head sees keys 0 .. its position; one
    # multiply-add each in Q K^T and in P V (4 flops per key per dimension)
    ql = step.query_lens.to(torch.float64)
    ctx = step.context_lens.to(torch.float64)
    visible = float((ql * ctx + ql * (ql + 1) / 2).sum())
    flops = 4.0 * d * H * visible
    return {"attention": attn, "kv_write": kvw, "kv_unique": kv_unique, "kv_logical": kv_logical,
            "step": attn + kvw, "flops": flops}


def shared_prefix_blocks(step: wl.Step) -> int:
    """Leading table blocks every request shares with request 0 (what a prefix
    cache knows when it hands out the blocks), bounded by every request's
    context; 0 when fewer than two requests or nothing is shared."""
    if step.num_seqs < 2:
        return 0
    t = step.block_tables
    same = (t == t[0:1]).all(dim=0).tolist()
    k = 0
    while k < len(same) and same[k]:
        k += 1
    ctx_min = int(step.context_lens.min())
    return min(k, ctx_min // step.block_size)


def has_prefill(step: wl.Step) -> bool:
    """Does the call run the tensor-core chunk kernel (some request with more
    than 64 rows q_r * G, and a head layout with a tensor-core tile)?"""
    G = step.num_q_heads // step.num_kv_heads
    tile_ok = step.head_size in (64, 128) and 128 % G == 0
    return tile_ok and step.max_query_len * G > 64


def decode_self_planned(step: wl.Step, prefix_blocks: int, fp8: bool, sms: int) -> bool:
    """The library's rule (paged_attn.cu, decode_self_plan_ok) for a call whose
    decode kernel plans itself, so that no plan kernel runs: every request a
    split row, nothing else on the call, automatic splits, and a batch small
    for the decode grid (its warps less the last CTA's)."""
    G = step.num_q_heads // step.num_kv_heads
    per_sm = {(64, False): 4, (128, False): 2, (64, True): 3, (128, True): 2}[(step.head_size, fp8)]
    resident = sms * per_sm
    pages = -(-step.max_seq_len // step.block_size)
    splits = max(1, min(pages, 32))
    max_chunks = step.num_seqs * splits + -(-(step.num_tokens * G) // 16) + step.num_seqs
    max_items = max_chunks * step.num_kv_heads
    warps = max(1, min(resident - 1, -(-max_items // 4))) * 4
    return (not has_prefill(step) and resident >= 2 and prefix_blocks == 0 and 1 <= step.num_seqs <= 1024
            and step.max_query_len * G <= 16 and step.num_seqs * step.num_kv_heads <= warps
            and step.num_seqs * pages * step.num_kv_heads <= 24 * warps)


def launches_per_step(step: wl.Step, prefix_blocks: int, fp8: bool, sms: int) -> int:
    """Kernels of one layer-step: kv_write, plan (not when the decode kernel
    plans the call itself), decode, combine; the prefill kernel when some
    request has more than 64 rows; the shared-prefix kernel when asked for."""
    G = step.num_q_heads // step.num_kv_heads
    tile_ok = step.head_size in (64, 128) and 128 % G == 0
    n = 3 if decode_self_planned(step, prefix_blocks if tile_ok else 0, fp8, sms) else 4
    if has_prefill(step):
        n += 1
    if tile_ok and prefix_blocks > 0:
        n += 1
    return n


FALLBACK_BF16_TFLOPS = 1900.0


def peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured (MEASURED_PEAKS.json: burst copy, burst cuBLAS bf16)"}
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS, "source": "fallback"}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() in ("active", "1"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def replica_seed(workload: str, rank: int) -> int:
    """Each rank runs its own replica of the batch: same shape, its own draws."""
    return wl.seed_of(workload) + 1000 * rank


def max_over_ranks(values, world: int, device=None):
    """Element-wise max of per-rank timings (the job takes as long as its
    slowest rank); the only cross-rank exchange of the benchmark."""
    if world <= 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def job_throughput(bytes_per_step_per_rank: float, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank moved its replica's bytes in the slowest rank's time."""
    return world * bytes_per_step_per_rank / (ms_per_step * 1e-3) / 1e9


def run_gpu(args, rank: int, world: int) -> dict:
    import paged_kv_cache_111_gb300 as pkv
    from paged_kv_cache_111_gb300 import _build
    _build.build()

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    step = wl.make_workload(args.workload, seed=replica_seed(args.workload, rank),
                            permute_blocks=not args.contiguous_blocks)
    if args.subset:
        # the first `subset` requests with a compact pool (profiling-size case)
        step = step.subset(list(range(min(args.subset, step.num_seqs))), name=f"{args.workload}[:{args.subset}]")
    T, H, d = step.num_tokens, step.num_q_heads, step.head_size
    to = {f: getattr(step, f).to(dev).contiguous() for f in
          ("seq_lens", "query_start_loc", "block_tables", "query", "key", "value", "slot_mapping")}
    fp8 = args.kv_dtype == "fp8"
    scales = fp8_scales(step) if fp8 else None
    if fp8:
        pool = torch.full(step.pool_shape(), 0x7F, dtype=torch.uint8, device=dev)   # E4M3 NaN
    else:
        pool = wl.make_poisoned_pool_like(step, device=dev)

    def write(key, value, slots):
        if fp8:
            pkv.kv_write_fp8(pool, key, value, slots, scales[0], scales[1])
        else:
            pkv.kv_write(pool, key, value, slots)

    hk, hv, hs = step.hist_key, step.hist_value, step.hist_slot_mapping
    chunk = 1 << 16
    for a in range(0, hs.numel(), chunk):
        b = min(hs.numel(), a + chunk)
        write(hk[a:b].to(dev), hv[a:b].to(dev), hs[a:b].to(dev))
    del hk, hv
    K = shared_prefix_blocks(step) if args.shared_prefix_blocks < 0 else args.shared_prefix_blocks
    if K:
        ws_bytes = pkv.paged_attn_shared_prefix_workspace_size(step.num_seqs, T, step.max_query_len,
                                                               step.max_seq_len, H, step.num_kv_heads, d, K)
    else:
        ws_bytes = pkv.paged_attn_workspace_size(step.num_seqs, T, step.max_query_len, step.max_seq_len, H,
                                                 step.num_kv_heads, d)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    out = torch.empty(T, H, d, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)
    maxq, maxs = step.max_query_len, step.max_seq_len

    def attention(q, tables, lens, qsl):
        if fp8 and K:
            pkv.paged_attn_shared_prefix_fp8(out, q, pool, tables, lens, qsl, maxq, maxs, step.scale, scales[0],
                                             scales[1], K, ws)
        elif fp8:
            pkv.paged_attn_fp8(out, q, pool, tables, lens, qsl, maxq, maxs, step.scale, scales[0], scales[1], ws)
        elif K:
            pkv.paged_attn_shared_prefix(out, q, pool, tables, lens, qsl, maxq, maxs, step.scale, K, ws)
        else:
            pkv.paged_attn(out, q, pool, tables, lens, qsl, maxq, maxs, step.scale, ws)

    def one_step(ev=(None, None, None, None)):
        """kv_write, paged_attn, combine; ev[k] (if not None) is recorded before
        call k and ev[3] after the last."""
        if ev[0] is not None:
            ev[0].record(stream)
        write(to["key"], to["value"], to["slot_mapping"])
        if ev[1] is not None:
            ev[1].record(stream)
        attention(to["query"], to["block_tables"], to["seq_lens"], to["query_start_loc"])
        if ev[2] is not None:
            ev[2].record(stream)
        pkv.paged_attn_combine(out, ws)
        if ev[3] is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize(dev)
    status = pkv.workspace_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {pkv.STATUS_NAMES.get(status, status)}")

    graph = None
    if args.graph:
        # the whole layer-step captured once and replayed: no host work per step
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            one_step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize(dev)
        stream = torch.cuda.current_stream(dev)

    # Inputs that fit in L2 would stay cached from one step to the next: for
    # such workloads every timed step starts from a cold L2 (a buffer of twice
    # the L2 size is written, then another one read, so that no dirty line of
    # the flush is written back during the step), and steps are timed one by
    # one with events around each step only.
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (129 << 20))
    ab_step = algorithmic_bytes(step, 1 if fp8 else 2)
    flush = ab_step["kv_unique"] <= 2 * l2_bytes
    flush_bufs = None
    if flush:
        n = (2 * l2_bytes + 3) // 4
        flush_bufs = (torch.empty(n, dtype=torch.float32, device=dev), torch.ones(n, dtype=torch.float32, device=dev))
        flush_sink = torch.empty((), dtype=torch.float32, device=dev)

    def cold_l2():
        flush_bufs[0].fill_(0.0)
        torch.sum(flush_bufs[1], dim=0, out=flush_sink)

    def run_steps(n_steps, phase_events):
        """Time n_steps steps on the device; returns (mean ms per step, phase ms or None,
        per-step ms or None)."""
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4 if phase_events else 2)]
              for _ in range(n_steps if (flush or phase_events) else 1)]
        if flush or phase_events:
            for i in range(n_steps):
                if flush:
                    cold_l2()
                e = ev[i]
                if graph is not None:
                    e[0].record(stream)
                    graph.replay()
                    e[-1].record(stream)
                else:
                    one_step(e if phase_events else (e[0], None, None, e[1]))
            torch.cuda.synchronize(dev)
            per = [e[0].elapsed_time(e[-1]) for e in ev]
            mean = sum(per) / n_steps
        else:
            per = None
            ev[0][0].record(stream)
            for _ in range(n_steps):
                if graph is not None:
                    graph.replay()
                else:
                    one_step()
            ev[0][1].record(stream)
            torch.cuda.synchronize(dev)
            mean = ev[0][0].elapsed_time(ev[0][1]) / n_steps
        if world > 1:
            torch.distributed.barrier()
        phases = None
        if phase_events and graph is None:
            phases = tuple(sum(e[k].elapsed_time(e[k + 1]) for e in ev) / n_steps for k in range(3))
        return mean, phases, per

    # The clock sampler runs from an untimed settle loop of the same step (at
    # least SETTLE_S seconds, so the record holds many samples taken under
    # this load) through the headline, phase and end-to-end passes.
    clk = ClockSampler(dev.index)
    clk.__enter__()
    t_settle = time.perf_counter() + SETTLE_S
    n_settle = 0
    while time.perf_counter() < t_settle:
        for _ in range(16):
            if graph is not None:
                graph.replay()
            else:
                one_step()
        n_settle += 16
        torch.cuda.synchronize(dev)
    # the headline: steps back to back (no event between the kernels of a step)
    step_ms, _, _ = run_steps(args.steps, False)
    total_ms = step_ms * args.steps
    # the phase breakdown (kv_write, paged_attn, combine), events between the calls
    if graph is None:
        _, (kvw_ms, attn_ms, comb_ms), phase_per = run_steps(min(args.steps, 300), True)
    else:
        # one graph per step: the phases are not separable; attribute the step
        kvw_ms = comb_ms = float("nan")
        attn_ms = step_ms
        phase_per = None
    status = pkv.workspace_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {pkv.STATUS_NAMES.get(status, status)}")

    # ---- end to end through the public API with host buffers ----------------
    # The step's inputs sit in one pinned host buffer (each tensor 256-byte
    # aligned in it), as an engine stages a step's metadata and activations,
    # and travel in one copy per step; the calls take views of its device copy.
    fields = ("seq_lens", "query_start_loc", "block_tables", "query", "key", "value", "slot_mapping")
    src = {f: getattr(step, f).contiguous() for f in fields}
    offs, n_bytes = {}, 0
    for f in fields:
        offs[f] = n_bytes
        n_bytes += (src[f].numel() * src[f].element_size() + 255) // 256 * 256
    host_buf = torch.empty(n_bytes, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(n_bytes, dtype=torch.uint8, device=dev)

    def view_of(buf, f):
        t = src[f]
        return buf[offs[f]:offs[f] + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    for f in fields:
        view_of(host_buf, f).copy_(src[f])
    dev_in = {f: view_of(dev_buf, f) for f in fields}
    host_out = torch.empty(T, H, d, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in src.values())
    d2h = host_out.numel() * host_out.element_size()
    e2e_steps = max(3, min(args.steps, 200)) if args.e2e else 0

    def e2e_step():
        dev_buf.copy_(host_buf, non_blocking=True)
        write(dev_in["key"], dev_in["value"], dev_in["slot_mapping"])
        attention(dev_in["query"], dev_in["block_tables"], dev_in["seq_lens"], dev_in["query_start_loc"])
        pkv.paged_attn_combine(out, ws)
        host_out.copy_(out, non_blocking=True)

    e2e_ms = float("nan")
    if e2e_steps:
        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        if flush:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(e2e_steps)]
            for e0, e1 in ev:
                cold_l2()
                e0.record(stream)
                e2e_step()
                e1.record(stream)
            torch.cuda.synchronize(dev)
            e2e_ms = sum(e0.elapsed_time(e1) for e0, e1 in ev) / e2e_steps
        else:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(e2e_steps):
                e2e_step()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            e2e_ms = e0.elapsed_time(e1) / e2e_steps

    clk.__exit__(None, None, None)
    clocks = clk.summary()
    clocks["window"] = (f"untimed settle loop of {n_settle} steps (>= {SETTLE_S:g} s), then the headline, phase "
                        f"and end-to-end passes")

    # ---- same-run copy probe (device-to-device copy, read + write bytes) ------
    # and a read-only probe (a sum over a 4 GiB buffer: read bytes only)
    probe_gbs = read_gbs = None
    if args.copy_probe:
        n = 1 << 30
        a = torch.empty(n, dtype=torch.bfloat16, device=dev)
        b = torch.empty_like(a)
        a.fill_(1.0)
        best = math.inf
        for _ in range(10):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            b.copy_(a)
            s1.record(stream)
            torch.cuda.synchronize(dev)
            best = min(best, s0.elapsed_time(s1))
        probe_gbs = 2 * n * 2 / (best * 1e-3) / 1e9
        del a, b
        x = torch.ones(1 << 30, dtype=torch.float32, device=dev)
        acc = torch.empty((), dtype=torch.float32, device=dev)
        best = math.inf
        for _ in range(10):
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            torch.sum(x, dim=0, out=acc)
            s1.record(stream)
            torch.cuda.synchronize(dev)
            best = min(best, s0.elapsed_time(s1))
        read_gbs = x.numel() * 4 / (best * 1e-3) / 1e9
        del x

    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return {"step": step, "shared_prefix_blocks": K,
            "launches_per_step": launches_per_step(step, K, args.kv_dtype == "fp8", sms),
            "fp8_scales": scales,
            "total_ms": total_ms, "kvw_ms": kvw_ms, "attn_ms": attn_ms, "comb_ms": comb_ms,
            "phase_step_ms": phase_per,
            "e2e_ms": e2e_ms, "h2d": h2d, "d2h": d2h, "clocks": clocks, "probe_gbs": probe_gbs,
            "read_probe_gbs": read_gbs,
            "l2_flush": flush, "l2_bytes": l2_bytes}


# ---------------------------------------------------------------------------
# the oracle on host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

def oracle_sample(step: wl.Step, n_req: int, seed: int) -> wl.Step:
    g = torch.Generator().manual_seed(seed)
    idx = torch.randperm(step.num_seqs, generator=g)[:max(1, min(n_req, step.num_seqs))]
    return step.subset(sorted(idx.tolist()))


def time_oracle_step(sub: wl.Step, fp8_scales=None, num_threads: int = 0) -> dict:
    """One oracle step on ``sub``: cache write of the new tokens, then
    attention (over an E4M3 cache when fp8_scales = (k_scale, v_scale) is
    given), on num_threads host threads (0: all), each phase timed on its own.
    Returns {"s", "kv_write_s", "attention_s", "bytes", "threads"} (bytes: the
    sample's algorithmic bytes of the whole step)."""
    import oracle
    if fp8_scales is None:
        cache = oracle.new_cache(sub.num_blocks, sub.num_kv_heads, sub.head_size)
        oracle.kv_write(cache, sub.hist_key, sub.hist_value, sub.hist_slot_mapping)
        t0 = time.perf_counter()
        oracle.kv_write(cache, sub.key, sub.value, sub.slot_mapping)
        t1 = time.perf_counter()
        oracle.paged_attn(cache, sub.query, sub.block_tables, sub.seq_lens, sub.query_start_loc,
                          sub.num_q_heads, sub.scale, num_threads)
        t2 = time.perf_counter()
        nbytes = algorithmic_bytes(sub)["step"]
    else:
        ks, vs = fp8_scales
        cache = oracle.new_cache_fp8(sub.num_blocks, sub.num_kv_heads, sub.head_size)
        oracle.kv_write_fp8(cache, sub.hist_key, sub.hist_value, sub.hist_slot_mapping, ks, vs)
        t0 = time.perf_counter()
        oracle.kv_write_fp8(cache, sub.key, sub.value, sub.slot_mapping, ks, vs)
        t1 = time.perf_counter()
        oracle.paged_attn_fp8(cache, sub.query, sub.block_tables, sub.seq_lens, sub.query_start_loc,
                              sub.num_q_heads, sub.scale, ks, vs, num_threads)
        t2 = time.perf_counter()
        nbytes = algorithmic_bytes(sub, 1)["step"]
    return {"s": t2 - t0, "kv_write_s": t1 - t0, "attention_s": t2 - t1, "bytes": nbytes,
            "threads": num_threads or oracle.max_threads()}


def phase_summary(runs) -> dict:
    """Mean ms per sampled step of each phase over a list of time_oracle_step results."""
    n = len(runs)
    return {"kv_write": sum(r["kv_write_s"] for r in runs) / n * 1e3,
            "attention": sum(r["attention_s"] for r in runs) / n * 1e3,
            "total": sum(r["s"] for r in runs) / n * 1e3}


def fp8_scales(step: wl.Step):
    """Per-tensor E4M3 scales from the step's own K and V (largest magnitude / 448),
    as a calibration pass would set them; rounded to fp32."""
    def amax(*ts):
        return max(float(t.float().abs().max()) if t.numel() else 0.0 for t in ts)
    ks = max(amax(step.hist_key, step.key), 1e-30) / 448.0
    vs = max(amax(step.hist_value, step.value), 1e-30) / 448.0
    return float(np.float32(ks)), float(np.float32(vs))


def cpu_baseline(step: wl.Step, budget_s: float = 10.0, scales=None) -> dict:
    import oracle
    oracle.build()
    n_req = max(1, step.num_seqs // 4)
    sub = oracle_sample(step, n_req, 7)
    runs = []
    t_end = time.perf_counter() + budget_s
    while len(runs) < 3 or time.perf_counter() < t_end:
        runs.append(time_oracle_step(sub, scales))
        if len(runs) >= 50:
            break
    ph = phase_summary(runs)
    nbytes, threads = runs[0]["bytes"], runs[0]["threads"]
    # the same oracle on one host thread, on a smaller sample (a sixteenth of the requests)
    sub1 = oracle_sample(step, max(1, step.num_seqs // 16), 8)
    runs1 = []
    t_end = time.perf_counter() + budget_s / 2
    while len(runs1) < 2 or time.perf_counter() < t_end:
        runs1.append(time_oracle_step(sub1, scales, num_threads=1))
        if len(runs1) >= 20:
            break
    ph1 = phase_summary(runs1)
    return {"value": nbytes / (ph["total"] * 1e-3) / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{sub.num_seqs} of {step.num_seqs} requests ({sub.num_tokens} query tokens), "
                      f"{len(runs)} timed oracle steps (cache write, then attention), mean {ph['total']:.1f} ms",
            "ms_per_sampled_step": ph,
            "tokens_per_s": sub.num_tokens / (ph["total"] * 1e-3),
            "single_thread": {"value": runs1[0]["bytes"] / (ph1["total"] * 1e-3) / 1e9, "unit": "GB/s", "cores": 1,
                              "ms_per_sampled_step": ph1,
                              "sample": f"{sub1.num_seqs} of {step.num_seqs} requests, {len(runs1)} timed oracle "
                                        f"steps, mean {ph1['total']:.1f} ms"}}


def run_reference(args, rank: int, world: int) -> None:
    if rank != 0:
        return
    import oracle
    oracle.build()
    step = wl.make_workload(args.workload)
    # size one step's sample so that warmup + steps finish in about two minutes
    probe = oracle_sample(step, 4, 11)
    dt = time_oracle_step(probe)["s"]
    per_req = max(dt / probe.num_seqs, 1e-4)
    budget_step = 120.0 / max(1, args.steps + args.warmup)
    n_req = int(max(1, min(step.num_seqs, budget_step / per_req)))
    samples = [oracle_sample(step, n_req, 100 + i) for i in range(min(4, args.steps + args.warmup))]
    for i in range(args.warmup):
        time_oracle_step(samples[i % len(samples)])
    runs = []
    tot_tok = 0
    for i in range(args.steps):
        s = samples[i % len(samples)]
        runs.append(time_oracle_step(s))
        tot_tok += s.num_tokens
    tot_t = sum(r["s"] for r in runs)
    tot_b = sum(r["bytes"] for r in runs)
    threads = runs[0]["threads"]
    ph = phase_summary(runs)
    value = tot_b / tot_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "sample_requests_per_step": n_req},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{n_req} of {step.num_seqs} requests per step, {args.steps} steps"},
        "us_per_step": {"kv_write": ph["kv_write"] * 1e3, "paged_attn": ph["attention"] * 1e3,
                        "total": ph["total"] * 1e3},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "tokens_per_s": tot_tok / tot_t,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------

def traffic_key(step: wl.Step, fp8: bool, prefix_blocks: int) -> str:
    """Which kernels the attention call runs (the key of TRAFFIC)."""
    kind = "decode"
    if prefix_blocks:
        kind = "cascade"
    elif has_prefill(step):
        kind = "prefill"
    return ("e4m3 " if fp8 else "bf16 ") + kind


def traffic_of(key: str, ab: dict):
    """(DRAM bytes per call, where the ratio comes from) for the call's kernels,
    or (None, why) when no capture of the current sources covers them."""
    t = TRAFFIC.get(key)
    if not t or t["ratio"] is None:
        return None, f"no ncu capture of the {key} call"
    if attention_sources_hash() != t["sources_sha256_16"]:
        return None, f"kernel sources changed since the {key} capture"
    return t["ratio"] * ab["attention"], t["source"] + " (ratio scaled by this call's algorithmic bytes)"


def roofline(ab: dict, attn_ms: float, pk: dict, traffic_key: str) -> dict:
    """Roofline of the paged_attn call: HBM-bound (decode) unless its
    algorithmic flops at the tensor peak take longer than its bytes at the
    HBM peak (a prefill chunk), then tensor-bound."""
    t = attn_ms * 1e-3
    hbm_s = ab["attention"] / (pk["hbm_gbs"] * 1e9)
    tensor_s = ab["flops"] / (pk["bf16_tflops"] * 1e12)
    if tensor_s > hbm_s:
        ach = ab["flops"] / t / 1e12
        return {"bound": "tensor", "kernel": "paged_attn (plan + decode + tcgen05 prefill kernels)",
                "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": ach / pk["bf16_tflops"],
                "peak_source": pk["source"], "algorithmic_flops_per_launch": ab["flops"],
                "traffic": traffic_of(traffic_key, ab)[0], "traffic_source": traffic_of(traffic_key, ab)[1]}
    ach = ab["attention"] / t / 1e9
    traffic, why = traffic_of(traffic_key, ab)
    return {"bound": "hbm", "kernel": "paged_attn (plan + decode kernels)",
            "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": ach / pk["hbm_gbs"],
            "peak_source": pk["source"], "algorithmic_bytes_per_launch": ab["attention"],
            "traffic": traffic, "traffic_source": why}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="llama13b-decode", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-copy-probe", dest="copy_probe", action="store_false")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--graph", action="store_true",
                    help="capture the layer-step in a CUDA graph once and time its replays")
    ap.add_argument("--shared-prefix-blocks", type=int, default=-1,
                    help="cascade over this many shared leading table blocks (pkv_paged_attn_shared_prefix); "
                         "-1: the prefix every request's table shares with request 0's, 0: plain paged_attn")
    ap.add_argument("--contiguous-blocks", action="store_true",
                    help="hand out physical blocks in order (no random permutation): the cost-of-paging comparison")
    ap.add_argument("--kv-dtype", default="bf16", choices=["bf16", "fp8"],
                    help="cache element type: bf16, or E4M3 with per-tensor K/V scales (pkv_*_fp8)")
    ap.add_argument("--subset", type=int, default=0,
                    help="keep only the first N requests, with a compact pool (small profiling case)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", int(os.environ["LOCAL_RANK"])))
    r = run_gpu(args, rank, world)
    step = r["step"]
    fp8 = args.kv_dtype == "fp8"
    ab = algorithmic_bytes(step, 1 if fp8 else 2)
    ms_per_step = r["total_ms"] / args.steps
    ms_per_step, attn_max, e2e_max = max_over_ranks([ms_per_step, r["attn_ms"], r["e2e_ms"]], world,
                                                    device="cuda" if world > 1 else None)
    if rank != 0:
        torch.distributed.destroy_process_group()
        return
    pk = peaks()
    value = job_throughput(ab["step"], world, ms_per_step)
    attn_gbs = ab["attention"] / (r["attn_ms"] * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if fp8 else "bf16",
        "data": "synthetic",
        "config": {
            "workload": step.name, "num_seqs": step.num_seqs, "num_tokens": step.num_tokens,
            "num_q_heads": step.num_q_heads, "num_kv_heads": step.num_kv_heads, "head_size": step.head_size,
            "block_size": step.block_size, "num_blocks": step.num_blocks,
            "kv_bytes_per_step": ab["kv_unique"], "parallelism": f"replicas x{world}",
            "launch": "cuda graph replay" if args.graph else "eager",
            "shared_prefix_blocks": r["shared_prefix_blocks"],
            "physical_blocks": "in order" if args.contiguous_blocks else "random permutation",
            "kv_cache": (f"e4m3, k_scale {r['fp8_scales'][0]:.6g}, v_scale {r['fp8_scales'][1]:.6g}"
                         if fp8 else "bf16"),
            "l2": (f"flushed before every timed step (write then read {2 * r['l2_bytes'] >> 20} MiB); "
                   f"steps timed one by one" if r["l2_flush"] else
                   f"inputs larger than L2 ({ab['kv_unique'] / 1e6:.0f} MB of KV per step, L2 "
                   f"{r['l2_bytes'] / 1e6:.0f} MB), no flush; steps back to back"),
            "phases": "kv_write / paged_attn / combine from a separate pass with events between the calls",
        },
        "pct_of_peak": value / pk["hbm_gbs"],
        "tokens_per_s": world * step.num_tokens / (ms_per_step * 1e-3),
        "us_per_step": {k: (v * 1e3 if v == v else None) for k, v in
                        (("kv_write", r["kvw_ms"]), ("paged_attn", r["attn_ms"]), ("combine", r["comb_ms"]),
                         ("total", ms_per_step))},
        # the phase pass times each step on its own: its spread (events between the calls included)
        "phase_pass_step_us_p10_p50_p90": ([round(v * 1e3, 2) for v in percentiles(r["phase_step_ms"])]
                                           if r["phase_step_ms"] else None),
        "roofline": roofline(ab, r["attn_ms"], pk, traffic_key(step, fp8, r["shared_prefix_blocks"])),
        "copy_probe_gbs": r["probe_gbs"],
        "read_probe_gbs": r["read_probe_gbs"],
        # the call against the same run's probes: decode reads far more than it writes
        "attn_frac_of_probe": ({"copy": attn_gbs / r["probe_gbs"], "read_only": attn_gbs / r["read_probe_gbs"]}
                               if r["probe_gbs"] and r["read_probe_gbs"] else None),
        "e2e": ({"value": job_throughput(ab["step"], world, e2e_max), "unit": "GB/s",
                 "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": e2e_max}
                if e2e_max == e2e_max else None),
        "gpu_launches": r["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
    }
    if r["shared_prefix_blocks"]:
        line["roofline"]["kernel"] = line["roofline"]["kernel"].replace(
            "paged_attn (plan + decode", "paged_attn_shared_prefix (plan + decode + tcgen05 shared-prefix")
    if fp8:
        line["roofline"]["kernel"] = line["roofline"]["kernel"].replace(" decode", " E4M3 decode").replace(
            "tcgen05", "E4M3-widening tcgen05")
    if args.graph:
        line["roofline"]["kernel"] = "whole layer-step (kv_write + paged_attn + combine), CUDA-graph replay"
        line["roofline"]["traffic"] = None
        line["roofline"]["traffic_source"] = "graph replay: no per-call capture"
    if ab["kv_logical"] != ab["kv_unique"]:
        line["logical_kv_gbs_incl_l2_reuse"] = ab["kv_logical"] / (r["attn_ms"] * 1e-3) / 1e9
    if not args.no_cpu_baseline and world == 1:      # the oracle's baseline: rank 0 of a 1-GPU run only
        line["cpu_baseline"] = cpu_baseline(step, scales=r["fp8_scales"])
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

"""Seeded synthetic inputs for one paged-KV attention layer-step.

This module draws random numbers and lays out the step's inputs: request
lengths, the assignment of physical cache blocks, slot numbers, and bf16
query/key/value values. It computes nothing of the attention method itself.
Both the CUDA path and the CPU oracle take their inputs from here.

What a step contains follows the vLLM pages' statement of the problem:
new K/V tokens with a ``slot_mapping`` (each new token's physical slot,
``slot = block * block_size + offset``), per-request block tables that map
logical blocks to physical ones, ``seq_lens`` and ``query_start_loc`` for the
flattened batch, and a softmax scale ("Inside vLLM: Anatomy of a
High-Throughput LLM Inference System", section "Executing the forward pass":
slot_mapping and the flattened super-sequence; "continuous batching and
PagedAttention" tutorial, section 3.3 "Data structures").

Conventions of the inputs made here:

* ``seq_lens[r]`` counts every token of request r after this step's new
  tokens are written; the request's context is ``seq_lens[r] - query_len``.
* Padding slots are ``-1``.  Block-table entries past a request's last block
  are ``-1`` and are never read.
* The pool starts as bf16 NaN (0x7FC0) everywhere: a slot that no one wrote
  must never reach an output.
* The already-cached tokens ("history") are returned as a flat list of
  (key, value, slot) entries; each side places them in its own pool with its
  own kv_write before the step.

Random draws: one ``torch.Generator`` seeded per workload draws the lengths
and then the block permutation; the bulk N(0, 1) values (history K, history
V, new Q, new K, new V) come from per-chunk generators seeded from the
workload seed, a tag per tensor and the chunk index.
"""

from __future__ import annotations

import dataclasses
import functools
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional, Sequence

import torch

BLOCK_SIZE = 16
BF16_NAN_BITS = 0x7FC0


@dataclasses.dataclass
class Step:
    """One layer-step of synthetic inputs, all tensors on the CPU."""

    name: str
    num_q_heads: int
    num_kv_heads: int
    head_size: int
    num_blocks: int
    block_size: int
    scale: float                     # an fp32 value (stored as a Python float)
    seq_lens: torch.Tensor           # int32 [S]
    query_start_loc: torch.Tensor    # int32 [S+1]
    block_tables: torch.Tensor       # int32 [S, max_blocks_per_seq], -1 unused
    query: torch.Tensor              # bf16 [T, H, d]
    key: torch.Tensor                # bf16 [T, Hkv, d]
    value: torch.Tensor              # bf16 [T, Hkv, d]
    slot_mapping: torch.Tensor       # int64 [T]
    hist_key: torch.Tensor           # bf16 [C, Hkv, d]
    hist_value: torch.Tensor         # bf16 [C, Hkv, d]
    hist_slot_mapping: torch.Tensor  # int64 [C]
    # hist_index[r] lists, in position order, which history entries hold
    # positions 0 .. context-1 of request r (shared prefixes repeat entries).
    hist_index: List[torch.Tensor]
    description: str = ""

    # ---- sizes -----------------------------------------------------------
    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.numel())

    @property
    def num_tokens(self) -> int:
        return int(self.query.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def query_lens(self) -> torch.Tensor:
        return (self.query_start_loc[1:] - self.query_start_loc[:-1]).to(torch.int64)

    @property
    def context_lens(self) -> torch.Tensor:
        return self.seq_lens.to(torch.int64) - self.query_lens

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max().item()) if self.num_seqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.num_seqs else 0

    def pool_shape(self):
        """Pool layout: [num_blocks][num_kv_heads][2 (K, V)][block_size][head_size]."""
        return (self.num_blocks, self.num_kv_heads, 2, self.block_size, self.head_size)

    def pool_bytes(self) -> int:
        return (self.num_blocks * self.num_kv_heads * 2 * self.block_size
                * self.head_size * 2)

    def request_kv(self, r: int):
        """Contiguous (K, V) of request r, [seq_len, Hkv, d] bf16, in position order.

        Built from the generator's own record of which drawn values hold which
        position; it does not read any cache pool.
        """
        idx = self.hist_index[r]
        q0 = int(self.query_start_loc[r])
        q1 = int(self.query_start_loc[r + 1])
        k = torch.cat([self.hist_key[idx], self.key[q0:q1]], dim=0)
        v = torch.cat([self.hist_value[idx], self.value[q0:q1]], dim=0)
        return k, v

    def subset(self, requests: Sequence[int], name: Optional[str] = None) -> "Step":
        """The same step restricted to ``requests``, with physical blocks renumbered compactly.

        Blocks are renumbered in order of first appearance in the chosen
        requests' tables; the pool shrinks to those blocks.  Values are
        unchanged, so each chosen request sees exactly the same keys, values
        and queries as before.
        """
        requests = [int(r) for r in requests]
        B = self.block_size
        used_blocks: List[int] = []
        seen = set()
        for r in requests:
            nb = (int(self.seq_lens[r]) + B - 1) // B
            for b in self.block_tables[r, :nb].tolist():
                if b not in seen:
                    seen.add(b)
                    used_blocks.append(b)
        nb_new = max(1, len(used_blocks))
        lut = torch.full((self.num_blocks,), -1, dtype=torch.int64)
        if used_blocks:
            lut[torch.tensor(used_blocks, dtype=torch.int64)] = torch.arange(len(used_blocks))

        def relabel_slots(slots: torch.Tensor) -> torch.Tensor:
            blk = torch.div(slots, B, rounding_mode="floor")
            new_blk = lut[blk.clamp(min=0)]
            out = new_blk * B + (slots - blk * B)
            return torch.where((slots >= 0) & (new_blk >= 0), out, torch.full_like(out, -1))

        max_nb = max([(int(self.seq_lens[r]) + B - 1) // B for r in requests] + [1])
        tables = torch.full((len(requests), max_nb), -1, dtype=torch.int32)
        seq_lens = torch.zeros(len(requests), dtype=torch.int32)
        qsl = [0]
        q_rows, hist_index = [], []
        for i, r in enumerate(requests):
            nb = (int(self.seq_lens[r]) + B - 1) // B
            tables[i, :nb] = lut[self.block_tables[r, :nb].to(torch.int64)].to(torch.int32)
            seq_lens[i] = self.seq_lens[r]
            q0, q1 = int(self.query_start_loc[r]), int(self.query_start_loc[r + 1])
            q_rows.append(torch.arange(q0, q1))
            qsl.append(qsl[-1] + (q1 - q0))
            hist_index.append(self.hist_index[r])
        q_rows_t = torch.cat(q_rows) if q_rows else torch.zeros(0, dtype=torch.int64)
        # every history entry a chosen request references lives in a chosen
        # block (shared blocks hold the same tokens for every sharer)
        if hist_index and sum(h.numel() for h in hist_index):
            keep_idx = torch.unique(torch.cat(hist_index))
        else:
            keep_idx = torch.zeros(0, dtype=torch.int64)
        hist_lut = torch.full((self.hist_slot_mapping.numel(),), -1, dtype=torch.int64)
        hist_lut[keep_idx] = torch.arange(keep_idx.numel())
        new_hist_index = [hist_lut[h] for h in hist_index]
        return Step(
            name=name or f"{self.name}[subset]",
            num_q_heads=self.num_q_heads, num_kv_heads=self.num_kv_heads,
            head_size=self.head_size, num_blocks=nb_new, block_size=B, scale=self.scale,
            seq_lens=seq_lens, query_start_loc=torch.tensor(qsl, dtype=torch.int32),
            block_tables=tables,
            query=self.query[q_rows_t].contiguous(), key=self.key[q_rows_t].contiguous(),
            value=self.value[q_rows_t].contiguous(),
            slot_mapping=relabel_slots(self.slot_mapping[q_rows_t]),
            hist_key=self.hist_key[keep_idx].contiguous(),
            hist_value=self.hist_value[keep_idx].contiguous(),
            hist_slot_mapping=relabel_slots(self.hist_slot_mapping[keep_idx]),
            hist_index=new_hist_index,
            description=f"subset of {self.name}: requests {requests[:8]}{'...' if len(requests) > 8 else ''}",
        )


# ---------------------------------------------------------------------------
# drawing helpers
# ---------------------------------------------------------------------------

_CHUNK = 1 << 22


def _chunk_seed(base: int, tag: int, chunk: int) -> int:
    """A 63-bit seed for one chunk of one bulk tensor (splitmix64 finaliser)."""
    z = (base * 0x9E3779B97F4A7C15 + tag * 0xBF58476D1CE4E5B9 + chunk * 0x94D049BB133111EB) & (2**64 - 1)
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & (2**64 - 1)
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & (2**64 - 1)
    z ^= z >> 31
    return z & (2**63 - 1)


def _randn_bf16(shape, base_seed: int, tag: int, threads: Optional[int] = None) -> torch.Tensor:
    """N(0, 1) fp32 draws rounded to bf16 (round-to-nearest-even).

    The tensor is cut into fixed chunks of 2**22 elements; chunk c draws from
    its own ``torch.Generator`` seeded from (base_seed, tag, c), so the values
    do not depend on how many threads draw them.
    """
    n = 1
    for s in shape:
        n *= int(s)
    out = torch.empty(n, dtype=torch.bfloat16)
    nchunks = (n + _CHUNK - 1) // _CHUNK

    def work(c: int) -> None:
        m = min(_CHUNK, n - c * _CHUNK)
        g = torch.Generator().manual_seed(_chunk_seed(base_seed, tag, c))
        b = torch.empty(m, dtype=torch.float32)
        b.normal_(generator=g)
        out[c * _CHUNK:c * _CHUNK + m].copy_(b)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        workers = threads or min(16, os.cpu_count() or 1)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(work, range(nchunks)))
    return out.view(*shape)


def _fp32(x: float) -> float:
    return float(torch.tensor(x, dtype=torch.float32).item())


@dataclasses.dataclass
class RequestSpec:
    context_len: int
    query_len: int


def build_step(
    name: str,
    requests: Sequence[RequestSpec],
    num_q_heads: int,
    num_kv_heads: int,
    head_size: int,
    num_blocks: int,
    seed: int,
    *,
    shared_prefix_len: int = 0,
    shared_prefix_requests: Optional[Sequence[int]] = None,
    forks: Optional[Sequence[int]] = None,
    permute_blocks: bool = True,
    extra_table_cols: int = 0,
    scale: Optional[float] = None,
    gen: Optional[torch.Generator] = None,
    description: str = "",
) -> Step:
    """Lay out one step from per-request (context_len, query_len).

    ``shared_prefix_len`` (a multiple of the block size) tokens at the head of
    every request in ``shared_prefix_requests`` live in the same physical
    blocks (read-only sharing, reference count > 1 in the pages' sense).
    ``forks`` lists parent request indices: fork f is appended as a new
    request with the parent's lengths whose table equals the parent's except
    its last entry, a fresh block holding a copy of the parent's last block's
    cached tokens (copy-on-write of the last shared block).  Each fork draws
    its own new token(s).
    """
    B = BLOCK_SIZE
    if gen is None:
        gen = torch.Generator().manual_seed(seed)
    reqs = [RequestSpec(int(r.context_len), int(r.query_len)) for r in requests]
    forks = list(forks or [])
    share = set(shared_prefix_requests if shared_prefix_requests is not None
                else (range(len(reqs)) if shared_prefix_len else []))
    if shared_prefix_len % B:
        raise ValueError("shared prefix must be whole blocks")
    for f in forks:
        reqs.append(RequestSpec(reqs[f].context_len, reqs[f].query_len))
    S = len(reqs)
    seq_lens = [r.context_len + r.query_len for r in reqs]
    for i, r in enumerate(reqs):
        if r.context_len < 0 or r.query_len < 0:
            raise ValueError("negative length")
        if i in share and r.context_len < shared_prefix_len:
            raise ValueError("shared prefix longer than a request's context")

    # ---- block permutation ------------------------------------------------
    if permute_blocks:
        perm = torch.randperm(num_blocks, generator=gen).tolist()
    else:
        perm = list(range(num_blocks))
    cursor = 0

    def take(n: int) -> List[int]:
        nonlocal cursor
        if cursor + n > num_blocks:
            raise ValueError(f"pool of {num_blocks} blocks too small")
        out = perm[cursor:cursor + n]
        cursor += n
        return out

    n_prefix_blocks = shared_prefix_len // B
    prefix_blocks = take(n_prefix_blocks) if (n_prefix_blocks and share) else []
    tables: List[List[int]] = []
    n_base = S - len(forks)
    for i in range(n_base):
        nb = (seq_lens[i] + B - 1) // B
        if i in share and prefix_blocks:
            tables.append(prefix_blocks + take(nb - n_prefix_blocks))
        else:
            tables.append(take(nb))
    for fi, f in enumerate(forks):
        t = list(tables[f])
        if not t:
            raise ValueError("cannot fork an empty request")
        if len(t) - 1 < (n_prefix_blocks if f in share else 0):
            raise ValueError("fork would copy a shared-prefix block")
        t[-1] = take(1)[0]
        tables.append(t)
    max_nb = max([len(t) for t in tables] + [1]) + extra_table_cols
    block_tables = torch.full((S, max_nb), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        if t:
            block_tables[i, :len(t)] = torch.tensor(t, dtype=torch.int32)

    # ---- history: which (request, position) needs a drawn value -----------
    tab_t = [torch.tensor(t, dtype=torch.int64) for t in tables]

    def slots_of(i: int, j0: int, j1: int) -> torch.Tensor:
        j = torch.arange(j0, j1, dtype=torch.int64)
        return tab_t[i][torch.div(j, B, rounding_mode="floor")] * B + j % B

    slot_chunks: List[torch.Tensor] = []
    hist_index: List[torch.Tensor] = [torch.zeros(0, dtype=torch.int64) for _ in range(S)]
    n_drawn = 0
    prefix_entries = torch.zeros(0, dtype=torch.int64)
    if prefix_blocks:
        pb = torch.tensor(prefix_blocks, dtype=torch.int64)
        j = torch.arange(shared_prefix_len, dtype=torch.int64)
        slot_chunks.append(pb[j // B] * B + j % B)
        prefix_entries = torch.arange(shared_prefix_len, dtype=torch.int64)
        n_drawn = shared_prefix_len
    for i in range(n_base):
        start = 0
        parts = []
        if i in share and prefix_blocks:
            parts.append(prefix_entries)
            start = shared_prefix_len
        n = reqs[i].context_len - start
        if n > 0:
            slot_chunks.append(slots_of(i, start, reqs[i].context_len))
            parts.append(torch.arange(n_drawn, n_drawn + n, dtype=torch.int64))
            n_drawn += n
        if parts:
            hist_index[i] = torch.cat(parts)
    # forks: reuse the parent's entries; the copied last block gets duplicate
    # entries (same values, new slots)
    copy_chunks: List[torch.Tensor] = []
    n_total = n_drawn
    for fi, f in enumerate(forks):
        i = n_base + fi
        ctx = reqs[i].context_len
        last_blk_start = min((len(tables[i]) - 1) * B, ctx)
        src_e = hist_index[f][last_blk_start:ctx]
        copy_chunks.append(src_e)
        slot_chunks.append(slots_of(i, last_blk_start, ctx))
        hist_index[i] = torch.cat([hist_index[f][:last_blk_start],
                                   torch.arange(n_total, n_total + src_e.numel(), dtype=torch.int64)])
        n_total += src_e.numel()
    hist_slots = torch.cat(slot_chunks) if slot_chunks else torch.zeros(0, dtype=torch.int64)
    copy_src = torch.cat(copy_chunks) if copy_chunks else torch.zeros(0, dtype=torch.int64)

    hk = _randn_bf16((n_drawn, num_kv_heads, head_size), seed, 1)
    hv = _randn_bf16((n_drawn, num_kv_heads, head_size), seed, 2)
    if copy_src.numel():
        hk = torch.cat([hk, hk[copy_src]], dim=0)
        hv = torch.cat([hv, hv[copy_src]], dim=0)

    # ---- new tokens --------------------------------------------------------
    qsl = [0]
    new_chunks: List[torch.Tensor] = []
    for i, r in enumerate(reqs):
        new_chunks.append(slots_of(i, r.context_len, r.context_len + r.query_len))
        qsl.append(qsl[-1] + r.query_len)
    new_slots = torch.cat(new_chunks) if new_chunks else torch.zeros(0, dtype=torch.int64)
    T = qsl[-1]
    q = _randn_bf16((T, num_q_heads, head_size), seed, 3)
    k = _randn_bf16((T, num_kv_heads, head_size), seed, 4)
    v = _randn_bf16((T, num_kv_heads, head_size), seed, 5)

    return Step(
        name=name,
        num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_size=head_size,
        num_blocks=num_blocks, block_size=B,
        scale=_fp32(1.0 / math.sqrt(head_size)) if scale is None else _fp32(scale),
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32),
        query_start_loc=torch.tensor(qsl, dtype=torch.int32),
        block_tables=block_tables,
        query=q, key=k, value=v,
        slot_mapping=new_slots,
        hist_key=hk, hist_value=hv,
        hist_slot_mapping=hist_slots,
        hist_index=hist_index,
        description=description,
    )


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

WORKLOADS = {
    "tiny-decode": dict(
        id=1, text="tiny decode-only step: 4 requests, 8 q heads = 8 kv heads, head_size 64, "
                   "seq_len uniform in [1,128], 64-block pool assigned by a seeded permutation"),
    "tinyllama-decode": dict(
        id=2, text="TinyLlama-1.1B-shaped decode layer-step: 64 requests, 32 q / 4 kv heads (GQA 8), "
                   "head_size 64, seq_len uniform in [512,2048], 16384-block pool"),
    "llama13b-decode": dict(
        id=3, text="LLaMA-13B-shaped decode layer-step: 256 requests, 40 q = 40 kv heads, head_size 128, "
                   "seq_len lognormal (mean ~800, sigma 0.8) clipped to [16,4096], 100000-block pool"),
    "llama3-8b-mixed": dict(
        id=4, text="Llama-3-8B-shaped mixed chunked-prefill step: decodes at seq_len 700 and 1500, then a "
                   "2046-token first prefill chunk; 32 q / 8 kv heads, head_size 128, 16384-block pool"),
    "llama3-70b-prefix": dict(
        id=5, text="Llama-3-70B-shaped prefix-sharing decode layer-step: 64 requests sharing a 1024-token "
                   "prefix, private suffix uniform in [16,512], plus 8 forks sharing all but their last "
                   "block; 64 q / 8 kv heads, head_size 128, 200000-block pool"),
}


def seed_of(name: str) -> int:
    return 20260000 + WORKLOADS[name]["id"]


def make_workload(name: str, seed: Optional[int] = None, permute_blocks: bool = True) -> Step:
    """Build one of the named workloads (full size).

    ``permute_blocks=False`` hands out physical blocks in order (each
    request's pages contiguous in the pool), the same draws otherwise: the
    contiguous-cache comparison point for the cost of paging.
    """
    if name not in WORKLOADS:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}")
    seed = seed_of(name) if seed is None else seed
    gen = torch.Generator().manual_seed(seed)
    text = WORKLOADS[name]["text"]
    build_step = functools.partial(_build_step_any, permute_blocks=permute_blocks)
    if name == "tiny-decode":
        L = torch.randint(1, 129, (4,), generator=gen).tolist()
        reqs = [RequestSpec(l - 1, 1) for l in L]
        return build_step(name, reqs, 8, 8, 64, 64, seed, gen=gen, description=text)
    if name == "tinyllama-decode":
        L = torch.randint(512, 2049, (64,), generator=gen).tolist()
        reqs = [RequestSpec(l - 1, 1) for l in L]
        return build_step(name, reqs, 32, 4, 64, 16384, seed, gen=gen, description=text)
    if name == "llama13b-decode":
        sigma = 0.8
        mu = math.log(800.0) - sigma * sigma / 2.0
        z = torch.randn(256, generator=gen, dtype=torch.float64)
        L = torch.clamp(torch.round(torch.exp(mu + sigma * z)), 16, 4096).to(torch.int64).tolist()
        reqs = [RequestSpec(l - 1, 1) for l in L]
        return build_step(name, reqs, 40, 40, 128, 100000, seed, gen=gen, description=text)
    if name == "llama3-8b-mixed":
        # decodes first (the scheduler serves running requests first), then the chunk
        reqs = [RequestSpec(699, 1), RequestSpec(1499, 1), RequestSpec(0, 2046)]
        return build_step(name, reqs, 32, 8, 128, 16384, seed, gen=gen, description=text)
    if name == "llama3-70b-prefix":
        suffix = torch.randint(16, 513, (64,), generator=gen).tolist()
        reqs = [RequestSpec(1024 + s - 1, 1) for s in suffix]
        return build_step(name, reqs, 64, 8, 128, 200000, seed, gen=gen,
                          shared_prefix_len=1024, forks=list(range(8)), description=text)
    raise AssertionError(name)


def _build_step_any(*args, permute_blocks: bool = True, **kw) -> Step:
    return build_step(*args, permute_blocks=permute_blocks, **kw)


def make_poisoned_pool_like(step: Step, device=None) -> torch.Tensor:
    """A pool of the step's shape filled with bf16 NaN (bit pattern 0x7FC0)."""
    pool = torch.empty(step.pool_shape(), dtype=torch.int16, device=device)
    pool.fill_(BF16_NAN_BITS)
    return pool.view(torch.bfloat16)

"""The E4M3 (FP8) cache option on the GPU against the fp64 oracle.

* kv_write_fp8: bit-exact over the whole cache (untouched bytes keep the NaN
  poison 0x7F), for several scales, including values that saturate at 448 and
  negative values that round to zero;
* paged_attn_fp8 + paged_attn_combine: the oracle's attention over the same
  E4M3 codes (value * scale), within the attention tolerance
  |gpu - ref| <= 2e-3 + 1e-2 |ref|.  Quantisation is part of the method and
  both sides take the same codes, so the tolerance covers only the
  attention arithmetic, as for a bf16 cache.
"""

import zlib

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_111_gb300 as pkv
import workloads as wl
from gpu_path import to_dev
from tolerance import check_close

pytestmark = pytest.mark.gpu

E4M3_NAN = 0x7F


def custom(reqs, H, Hkv, d, seed=1, nb=None, **kw):
    specs = [wl.RequestSpec(c, q) for c, q in reqs]
    need = sum((c + q + 15) // 16 for c, q in reqs) + 8
    return wl.build_step("custom", specs, H, Hkv, d, nb or max(2 * need, 16), seed, **kw)


def gpu_fp8_cache(step, k_scale, v_scale, dev):
    cache = torch.full(step.pool_shape(), E4M3_NAN, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = dev["hist_slot_mapping"].shape[0]
    for a in range(0, C, 1 << 16):
        b = min(C, a + (1 << 16))
        pkv.kv_write_fp8(cache, dev["hist_key"][a:b], dev["hist_value"][a:b], dev["hist_slot_mapping"][a:b],
                         k_scale, v_scale, status)
    pkv.kv_write_fp8(cache, dev["key"], dev["value"], dev["slot_mapping"], k_scale, v_scale, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return cache


def run_fp8(step, k_scale, v_scale, num_splits=0):
    dev = to_dev(step)
    cache = gpu_fp8_cache(step, k_scale, v_scale, dev)
    n = pkv.paged_attn_workspace_size(step.num_seqs, step.num_tokens, step.max_query_len, step.max_seq_len,
                                      step.num_q_heads, step.num_kv_heads, step.head_size)
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
    out = torch.full((step.num_tokens, step.num_q_heads, step.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    pkv.paged_attn_fp8(out, dev["query"], cache, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                       step.max_query_len, step.max_seq_len, step.scale, k_scale, v_scale, ws,
                       num_splits=num_splits)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    return cache, out


SCALES = [(1.0, 1.0), (0.0173, 3.7), (0.001, 0.5)]     # the last saturates |K| > 0.448 at 448


@pytest.mark.parametrize("k_scale,v_scale", SCALES)
@pytest.mark.parametrize("name", ["tiny-decode", "llama3-8b-mixed"])
def test_kv_write_fp8_is_bit_exact_over_the_whole_cache(name, k_scale, v_scale):
    step = wl.make_workload(name)
    dev = to_dev(step)
    cache = gpu_fp8_cache(step, k_scale, v_scale, dev)
    ref = oracle.new_cache_fp8(step.num_blocks, step.num_kv_heads, step.head_size)
    oracle.kv_write_fp8(ref, step.hist_key, step.hist_value, step.hist_slot_mapping, k_scale, v_scale)
    oracle.kv_write_fp8(ref, step.key, step.value, step.slot_mapping, k_scale, v_scale)
    got = cache.cpu().numpy()
    assert np.array_equal(got, ref), f"{int((got != ref).sum())} bytes differ"


def test_kv_write_fp8_signed_zero_saturation_and_padding():
    # hand-made rows: tiny negatives (round to -0), huge values (held at 448), padding slots
    T, Hkv, d = 4, 2, 64
    vals = torch.tensor([-1e-30, -2.0 ** -11, 2.0 ** -10, 3 * 2.0 ** -10, 1e4, -1e4, 447.9, 0.0], dtype=torch.float32)
    key = vals.repeat(T * Hkv * d // vals.numel()).reshape(T, Hkv, d).to(torch.bfloat16)
    value = (-key.float()).to(torch.bfloat16)
    slots = torch.tensor([3, -1, 17, 30], dtype=torch.int64)
    cache = torch.full((2, Hkv, 2, 16, d), E4M3_NAN, dtype=torch.uint8, device="cuda")
    pkv.kv_write_fp8(cache, key.cuda(), value.cuda(), slots.cuda(), 1.0, 1.0)
    ref = oracle.new_cache_fp8(2, Hkv, d)
    oracle.kv_write_fp8(ref, key, value, slots, 1.0, 1.0)
    assert np.array_equal(cache.cpu().numpy(), ref)


@pytest.mark.parametrize("name", ["tiny-decode", "tinyllama-decode", "llama3-70b-prefix"])
def test_attention_fp8_named_workloads(name):
    step = wl.make_workload(name)
    k_scale, v_scale = 0.0173, 0.031
    _, out = run_fp8(step, k_scale, v_scale)
    _, ref, _ = oracle.run_step_fp8(step, k_scale, v_scale)
    check_close(out, ref, f"{name} fp8")


def test_attention_fp8_mixed_step_with_a_long_chunk():
    step = wl.make_workload("llama3-8b-mixed")
    _, out = run_fp8(step, 1.0, 1.0)
    _, ref, _ = oracle.run_step_fp8(step, 1.0, 1.0)
    check_close(out, ref, "mixed fp8")


def test_attention_fp8_llama13b_every_row():
    """The 13B batch over an E4M3 cache, every output row against the
    oracle's attention over the same codes (pool compacted to the used
    blocks on the host)."""
    step = wl.make_workload("llama13b-decode")
    k_scale, v_scale = 0.02, 0.02
    _, out = run_fp8(step, k_scale, v_scale)
    out = out.cpu()
    sub = step.subset(range(step.num_seqs))
    assert torch.equal(sub.query, step.query)
    _, ref, _ = oracle.run_step_fp8(sub, k_scale, v_scale)
    check_close(out, ref, "llama13b fp8 every row")


EDGE = [
    ("page edges mha d64", [(0, 1), (14, 1), (15, 1), (16, 1), (30, 1), (31, 1), (32, 1)], 4, 4, 64, None),
    ("page edges gqa8 d128", [(0, 1), (14, 1), (15, 1), (16, 1), (30, 1), (31, 1), (32, 1)], 16, 2, 128, None),
    ("chunks and multi-token rows", [(5, 40), (17, 1), (0, 17), (33, 3), (100, 3)], 8, 2, 128, None),
    ("mqa G=32", [(70, 1), (3, 2), (0, 5)], 32, 1, 64, None),
    ("empty requests", [(20, 4), (0, 0), (47, 1), (5, 0)], 8, 4, 64, None),
    ("peaked softmax (scale 1.0)", [(300, 1), (50, 70)], 8, 2, 128, 1.0),
    ("prefix and forks", [(200, 1), (260, 1), (143, 1)], 16, 2, 128, None),
    ("8-row tiles q=4 G=2", [(50, 4), (3, 4), (400, 2)], 4, 2, 128, None),
]


@pytest.mark.parametrize("case", EDGE, ids=[c[0] for c in EDGE])
@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.0173, 3.7)])
def test_attention_fp8_edge_cases(case, k_scale, v_scale):
    name, reqs, H, Hkv, d, scale = case
    kw = {"shared_prefix_len": 64, "forks": [0, 2]} if name == "prefix and forks" else {}
    step = custom(reqs, H, Hkv, d, seed=zlib.crc32(name.encode()) % 1000, scale=scale, **kw)
    _, out = run_fp8(step, k_scale, v_scale)
    _, ref, _ = oracle.run_step_fp8(step, k_scale, v_scale)
    check_close(out, ref, f"{name} fp8")


@pytest.mark.parametrize("splits", [1, 3, 32])
def test_attention_fp8_forced_splits(splits):
    step = custom([(700, 1), (33, 1), (1500, 1), (255, 2)], 16, 2, 128, seed=40 + splits)
    _, out = run_fp8(step, 0.05, 0.05, num_splits=splits)
    _, ref, _ = oracle.run_step_fp8(step, 0.05, 0.05)
    check_close(out, ref, f"fp8 splits={splits}")


def test_attention_fp8_query_rows_of_very_different_magnitudes():
    # per-row power-of-two scaling of Q into f16: tiny and huge rows stay exact
    step = custom([(120, 1), (40, 2)], 8, 2, 128, seed=77)
    q = step.query.float()
    q[0, :4] *= 1e-20
    q[0, 4:] *= 3e4
    q[1, ::2] *= 1e6
    step.query = q.to(torch.bfloat16)
    step.scale = 1e-4
    _, out = run_fp8(step, 0.1, 0.1)
    _, ref, _ = oracle.run_step_fp8(step, 0.1, 0.1)
    check_close(out, ref, "fp8 extreme query rows")


def test_fp8_argument_errors():
    step = custom([(20, 1)], 4, 4, 64, seed=3)
    dev = to_dev(step)
    cache = torch.zeros(step.pool_shape(), dtype=torch.uint8, device="cuda")
    with pytest.raises(pkv.PagedKVError):
        pkv.kv_write_fp8(cache, dev["key"], dev["value"], dev["slot_mapping"], 0.0, 1.0)
    with pytest.raises(pkv.PagedKVError):
        pkv.kv_write_fp8(cache, dev["key"], dev["value"], dev["slot_mapping"], 1.0, float("nan"))
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    out = torch.empty(step.num_tokens, step.num_q_heads, step.head_size, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pkv.PagedKVError):
        pkv.paged_attn_fp8(out, dev["query"], cache, dev["block_tables"], dev["seq_lens"], dev["query_start_loc"],
                           step.max_query_len, step.max_seq_len, step.scale, -1.0, 1.0, ws)


def run_fp8_cascade(step, k_scale, v_scale, prefix_blocks, num_splits=0):
    dev = to_dev(step)
    cache = gpu_fp8_cache(step, k_scale, v_scale, dev)
    n = pkv.paged_attn_shared_prefix_workspace_size(step.num_seqs, step.num_tokens, step.max_query_len,
                                                    step.max_seq_len, step.num_q_heads, step.num_kv_heads,
                                                    step.head_size, prefix_blocks)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    out = torch.full((step.num_tokens, step.num_q_heads, step.head_size), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    pkv.paged_attn_shared_prefix_fp8(out, dev["query"], cache, dev["block_tables"], dev["seq_lens"],
                                     dev["query_start_loc"], step.max_query_len, step.max_seq_len, step.scale,
                                     k_scale, v_scale, prefix_blocks, ws, num_splits=num_splits)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 0
    return out


def test_attention_fp8_shared_prefix_workload_full_size():
    # 64 sharers of a 1024-token prefix plus forks: the prefix's E4M3 pages are
    # widened once per kv head for every sharer on the tensor-core kernel
    step = wl.make_workload("llama3-70b-prefix")
    out = run_fp8_cascade(step, 0.011, 0.009, 64)
    _, ref, _ = oracle.run_step_fp8(step, 0.011, 0.009)
    check_close(out, ref, "70b prefix cascade fp8")


@pytest.mark.parametrize("splits", [0, 3, 32])
def test_attention_fp8_shared_prefix_with_multi_token_rows(splits):
    specs = [wl.RequestSpec(300, 1), wl.RequestSpec(170, 2), wl.RequestSpec(520, 1), wl.RequestSpec(128, 2)]
    step = wl.build_step("fp8 cascade", specs, 16, 4, 64, 256, 71, shared_prefix_len=128)
    out = run_fp8_cascade(step, 0.02, 0.03, 8, num_splits=splits)
    _, ref, _ = oracle.run_step_fp8(step, 0.02, 0.03)
    check_close(out, ref, f"fp8 cascade splits={splits}")


@pytest.mark.parametrize("bad_request", [0, 1])
def test_fp8_out_of_pool_block_is_reported(bad_request):
    """A block id past the pool, in a decode row (request 0) or in a chunk on
    the widening tensor-core kernel (request 1), loads as zeros and is
    reported; the other request's rows are unaffected."""
    step = custom([(40, 1), (10, 150)], 8, 2, 128, seed=13)
    ks, vs = 0.011, 0.019
    dev = to_dev(step)
    cache = gpu_fp8_cache(step, ks, vs, dev)
    n = pkv.paged_attn_workspace_size(step.num_seqs, step.num_tokens, step.max_query_len, step.max_seq_len,
                                      8, 2, 128)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    bt = dev["block_tables"].clone()
    bt[bad_request, 2] = step.num_blocks + 1000
    out = torch.zeros(step.num_tokens, 8, 128, dtype=torch.bfloat16, device="cuda")
    pkv.paged_attn_fp8(out, dev["query"], cache, bt, dev["seq_lens"], dev["query_start_loc"], step.max_query_len,
                       step.max_seq_len, step.scale, ks, vs, ws)
    pkv.paged_attn_combine(out, ws)
    torch.cuda.synchronize()
    assert pkv.workspace_status(ws) == 7          # PKV_ERR_DEVICE_INDEX
    good = 1 - bad_request
    q0, q1 = int(step.query_start_loc[good]), int(step.query_start_loc[good + 1])
    _, ref, _ = oracle.run_step_fp8(step.subset([good]), ks, vs)
    check_close(out[q0:q1], ref, "request beside the bad block")


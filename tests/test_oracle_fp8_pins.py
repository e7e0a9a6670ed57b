"""Pins for the oracle's FP8 (E4M3) cache option, against things other than itself.

* the E4M3 code values against torch's own float8_e4m3fn type (all 256 codes);
* the encoder against torch's float32 -> float8_e4m3fn rounding (nearest, ties
  to even) on random, boundary and exact-midpoint values inside the range
  where torch does not overflow, and against a brute-force nearest-code search
  written here in numpy;
* the saturation and signed-zero closed forms;
* the FP8 cache write against torch's quotient-then-round on the same bytes,
  and its round-trip error bound (half a unit in the last place of E4M3);
* FP8 attention against the bf16 oracle on a bf16 cache that holds exactly the
  dequantised values (power-of-two scales make them exact in bf16), and
  against torch scaled_dot_product_attention in fp64 on contiguous dequantised
  K/V for arbitrary scales.
"""

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

F8 = torch.float8_e4m3fn


def torch_decode(codes: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(F8).to(torch.float64).numpy()


def torch_encode(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(F8).view(torch.uint8).numpy()


def oracle_encode(x: np.ndarray) -> np.ndarray:
    return np.array([oracle.e4m3_encode(float(v)) for v in np.asarray(x, dtype=np.float32)], dtype=np.uint8)


POS_CODES = np.arange(0, 0x7F, dtype=np.uint8)          # every finite non-negative code
POS_VALUES = torch_decode(POS_CODES)


def brute_force_code(x: float) -> int:
    """Nearest finite E4M3 code by search over all of them; ties to the even code."""
    a = abs(x)
    if a >= 448.0:
        c = 0x7E
    else:
        dist = np.abs(POS_VALUES - a)
        best = np.flatnonzero(dist == dist.min())
        c = int(best[0]) if len(best) == 1 else int([b for b in best if b % 2 == 0][0])
    return c | (0x80 if np.signbit(x) else 0)


def test_decode_matches_torch_on_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch_decode(codes)
    got = np.array([oracle.e4m3_decode(c) for c in codes])
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x38] == 1.0


def test_encode_matches_torch_rounding_inside_its_range():
    rng = np.random.default_rng(7)
    mids = (POS_VALUES[1:] + POS_VALUES[:-1]) / 2.0      # exact ties, all representable in fp32
    vals = np.concatenate([
        POS_VALUES, mids, np.nextafter(mids.astype(np.float32), np.float32(np.inf)).astype(np.float64),
        np.nextafter(mids.astype(np.float32), np.float32(-np.inf)).astype(np.float64),
        rng.standard_normal(20000) * np.exp2(rng.integers(-12, 9, 20000)),
        rng.uniform(440.0, 463.9, 200),
    ]).astype(np.float32)
    vals = vals[np.abs(vals) < 464.0]                    # torch overflows to NaN from 464 on
    vals = np.concatenate([vals, -vals])
    assert np.array_equal(oracle_encode(vals), torch_encode(vals))


def test_encode_matches_brute_force_search():
    rng = np.random.default_rng(11)
    vals = np.concatenate([rng.standard_normal(3000) * np.exp2(rng.integers(-11, 10, 3000)),
                           (POS_VALUES[1:] + POS_VALUES[:-1]) / 2.0, [0.0, 1000.0, 3.0e38]]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    got = oracle_encode(vals)
    ref = np.array([brute_force_code(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_saturation_and_signed_zero():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(464.0) == 0x7E
    # past the tie at 464 the nearest step up (480) is no E4M3 value: held at 448, never the NaN code
    for v in (464.5, 470.0, 479.0, 479.99, 480.0, 500.0):
        assert oracle.e4m3_encode(v) == 0x7E and oracle.e4m3_encode(-v) == 0xFE
    assert oracle.e4m3_encode(1.0e30) == 0x7E
    assert oracle.e4m3_encode(float("inf")) == 0x7E
    assert oracle.e4m3_encode(-float("inf")) == 0xFE
    assert oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(-2.0 ** -11) == 0x80       # rounds to zero, keeps its sign
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00        # tie between 0 and 2^-9: even code 0
    assert oracle.e4m3_encode(3 * 2.0 ** -10) == 0x02    # tie between codes 1 and 2: even code 2
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def small_step(seed=3, H=8, Hkv=2, d=64, reqs=((20, 1), (33, 2), (0, 17), (47, 1))):
    specs = [wl.RequestSpec(c, q) for c, q in reqs]
    need = sum((c + q + 15) // 16 for c, q in reqs) + 4
    return wl.build_step("fp8pin", specs, H, Hkv, d, need * 2, seed)


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.0173, 3.7), (0.25, 0.0625)])
def test_fp8_write_matches_torch_quotient_rounding(k_scale, v_scale):
    step = small_step()
    cache = oracle.new_cache_fp8(step.num_blocks, step.num_kv_heads, step.head_size)
    oracle.kv_write_fp8(cache, step.key, step.value, step.slot_mapping, k_scale, v_scale)
    ks = torch.tensor(k_scale, dtype=torch.float32)
    vs = torch.tensor(v_scale, dtype=torch.float32)
    qk = (step.key.float() / ks)
    qv = (step.value.float() / vs)
    assert qk.abs().max() < 464 and qv.abs().max() < 464  # inside torch's non-overflowing range
    ek = qk.to(F8).view(torch.uint8).numpy()
    ev = qv.to(F8).view(torch.uint8).numpy()
    touched = np.zeros(cache.shape[:1] + cache.shape[3:4], dtype=bool)
    for t, slot in enumerate(step.slot_mapping.tolist()):
        b, o = divmod(slot, 16)
        touched[b, o] = True
        assert np.array_equal(cache[b, :, 0, o, :], ek[t])
        assert np.array_equal(cache[b, :, 1, o, :], ev[t])
    # every other byte is still the NaN poison
    rest = cache.transpose(0, 3, 1, 2, 4)[~touched]
    assert (rest == oracle.E4M3_NAN).all()


def test_fp8_write_round_trip_error_is_within_half_an_ulp():
    step = small_step(seed=5, d=128)
    k_scale, v_scale = 0.05, 0.021
    cache = oracle.new_cache_fp8(step.num_blocks, step.num_kv_heads, step.head_size)
    oracle.kv_write_fp8(cache, step.key, step.value, step.slot_mapping, k_scale, v_scale)
    for t, slot in enumerate(step.slot_mapping.tolist()):
        b, o = divmod(slot, 16)
        for which, x, s in ((0, step.key[t], k_scale), (1, step.value[t], v_scale)):
            xq = x.double().numpy() / np.float64(np.float32(s))
            back = torch_decode(cache[b, :, which, o, :])
            a = np.abs(xq)
            # half-ulp of E4M3: 2^(e-4) for normal magnitudes, 2^-10 below 2^-6
            e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
            bound = np.exp2(e - 4) * (1 + 1e-6)
            assert (np.abs(back - np.clip(xq, -448.0, 448.0)) <= bound).all()


def dequantised_bf16_cache(cache8: np.ndarray, k_scale: float, v_scale: float) -> np.ndarray:
    """bf16 bit patterns of code * scale (exact when the scales are powers of two)."""
    vals = torch_decode(cache8.reshape(-1)).reshape(cache8.shape)
    vals[:, :, 0] *= k_scale
    vals[:, :, 1] *= v_scale
    t = torch.from_numpy(vals)
    b = t.to(torch.bfloat16)
    finite = torch.isfinite(t)
    assert torch.equal(b.double()[finite], t[finite])      # exact in bf16
    return b.view(torch.int16).numpy().view(np.uint16).copy()


@pytest.mark.parametrize("seed,H,Hkv,d", [(21, 8, 2, 64), (22, 16, 16, 128), (23, 32, 4, 128)])
def test_fp8_attention_equals_bf16_oracle_on_the_dequantised_cache(seed, H, Hkv, d):
    step = small_step(seed=seed, H=H, Hkv=Hkv, d=d, reqs=((40, 1), (3, 30), (17, 2), (64, 1)))
    k_scale, v_scale = 0.125, 4.0
    cache8, out8, lse8 = oracle.run_step_fp8(step, k_scale, v_scale)
    cache16 = dequantised_bf16_cache(cache8, k_scale, v_scale)
    out16, lse16 = oracle.paged_attn(cache16, step.query, step.block_tables, step.seq_lens,
                                     step.query_start_loc, step.num_q_heads, step.scale)
    assert np.array_equal(out8, out16) and np.array_equal(lse8, lse16)


@pytest.mark.parametrize("k_scale,v_scale", [(0.0173, 3.7), (1.0, 1.0)])
def test_fp8_attention_matches_torch_sdpa_on_contiguous_dequantised_kv(k_scale, v_scale):
    step = small_step(seed=31, H=16, Hkv=4, d=128, reqs=((50, 1), (0, 20), (31, 3)))
    _, out, _ = oracle.run_step_fp8(step, k_scale, v_scale)
    ref = torch.zeros(step.num_tokens, step.num_q_heads, step.head_size, dtype=torch.float64)
    ks = torch.tensor(k_scale, dtype=torch.float32)
    vs = torch.tensor(v_scale, dtype=torch.float32)
    for r in range(step.num_seqs):
        q0, q1 = int(step.query_start_loc[r]), int(step.query_start_loc[r + 1])
        L = int(step.seq_lens[r])
        c = L - (q1 - q0)
        k, v = step.request_kv(r)
        kd = (k.float() / ks).to(F8).to(torch.float64) * float(ks)
        vd = (v.float() / vs).to(F8).to(torch.float64) * float(vs)
        q = step.query[q0:q1].double().permute(1, 0, 2).unsqueeze(0)
        mask = torch.arange(L).unsqueeze(0) <= (c + torch.arange(q1 - q0).unsqueeze(1))
        o = torch.nn.functional.scaled_dot_product_attention(
            q, kd.permute(1, 0, 2).unsqueeze(0), vd.permute(1, 0, 2).unsqueeze(0), attn_mask=mask,
            scale=step.scale, enable_gqa=True)
        ref[q0:q1] = o[0].permute(1, 0, 2)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-12, atol=1e-12)

"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is a one-expression edit of ``oracle/pkv_oracle.c`` compiled
into a temporary library; the committed oracle is never modified.  For each
one, at least one of the pin tests in ``test_oracle_pins`` or
``test_oracle_fp8_pins`` must fail.
"""

import os
import subprocess
import sys

import pytest

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "pkv_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("gqa head mapping", "const int32_t g = h / G;", "const int32_t g = h % p->num_kv_heads;"),
    ("causal limit excludes self", "int64_t j1 = key_end < pos + 1 ? key_end : pos + 1;\n    for (int32_t e",
     "int64_t j1 = key_end < pos ? key_end : pos;\n    for (int32_t e"),
    ("causal limit one too far", "int64_t j1 = key_end < pos + 1 ? key_end : pos + 1;\n    for (int32_t e",
     "int64_t j1 = key_end < pos + 2 ? key_end : pos + 2;\n    for (int32_t e"),
    ("position ignores context", "const int64_t pos = context + i;", "const int64_t pos = i;"),
    ("keys read from the V half", "* cache_elem(p, phys, g, 0, (int32_t)(j % B), e)",
     "* cache_elem(p, phys, g, 1, (int32_t)(j % B), e)"),
    ("table indexed by offset", "const int32_t phys = table[j / B];\n        double dot",
     "const int32_t phys = table[j % B];\n        double dot"),
    ("offset taken as block index", "cache_elem(p, phys, g, 1, (int32_t)(j % B), e)",
     "cache_elem(p, phys, g, 1, (int32_t)((j / B) % B), e)"),
    ("scale dropped", "const double s = p->scale * dot;", "const double s = dot;"),
    ("no normalisation", "        out[e] /= z;\n    *lse = m + log(z);", "        out[e] /= 1.0;\n    *lse = m + log(z);"),
    ("lse without the maximum", "*lse = m + log(z);\n    if (weights)", "*lse = log(z);\n    if (weights)"),
    ("cache write offset", "/* padding token */\n        const int64_t block = slot / block_size;\n"
     "        const int32_t off = (int32_t)(slot % block_size);",
     "/* padding token */\n        const int64_t block = slot / block_size;\n"
     "        const int32_t off = (int32_t)((slot + 1) % block_size);"),
    ("fp8 cache write offset", "continue;\n        const int64_t block = slot / block_size;\n"
     "        const int32_t off = (int32_t)(slot % block_size);",
     "continue;\n        const int64_t block = slot / block_size;\n"
     "        const int32_t off = (int32_t)((slot + 1) % block_size);"),
    ("cache write K/V swapped", "memcpy(cache + cache_offset(block, h, 0, off, num_kv_heads, block_size, head_size),\n                   key + src",
     "memcpy(cache + cache_offset(block, h, 0, off, num_kv_heads, block_size, head_size),\n                   value + src"),
    ("combine ignores weights", "const double w = exp(part_lse[s] - m);", "const double w = 1.0;"),
    ("block copy covers one kv head", "const size_t block_elems = cache_offset(1, 0, 0, 0, num_kv_heads, block_size, head_size);",
     "const size_t block_elems = cache_offset(0, 1, 0, 0, num_kv_heads, block_size, head_size);"),
    ("e4m3 exponent bias", "v = ldexp(1.0 + m / 8.0, e - 7);", "v = ldexp(1.0 + m / 8.0, e - 8);"),
    ("e4m3 mantissa truncated", "const int m = (int)nearbyint((2.0 * fr - 1.0) * 8.0);",
     "const int m = (int)floor((2.0 * fr - 1.0) * 8.0);"),
    ("e4m3 subnormal step", "code = (int)nearbyint(ldexp(a, 9));", "code = (int)nearbyint(ldexp(a, 8));"),
    ("e4m3 ties away from zero", "const int m = (int)nearbyint((2.0 * fr - 1.0) * 8.0);",
     "const int m = (int)round((2.0 * fr - 1.0) * 8.0);"),
    ("e4m3 saturation threshold at 480", "if (a >= 448.0)\n        return sign | 0x7E;",
     "if (a >= 480.0)\n        return sign | 0x7E;"),
    ("e4m3 subnormal range one binade short", "if (a < ldexp(1.0, -6)) {", "if (a < ldexp(1.0, -7)) {"),
    ("slot 0 taken for padding", "if (slot < 0)\n            continue; /* padding token */",
     "if (slot <= 0)\n            continue; /* padding token */"),
    ("query row ignores its index", "const int64_t t = (int64_t)p->query_start_loc[r] + i;",
     "const int64_t t = (int64_t)p->query_start_loc[r];"),
    ("block copy reversed", "memcpy(cache + (size_t)dst * block_elems, cache + (size_t)src * block_elems,",
     "memcpy(cache + (size_t)src * block_elems, cache + (size_t)dst * block_elems,"),
    ("block copy of half a block", "               block_elems * sizeof(uint16_t));",
     "               block_elems / 2 * sizeof(uint16_t));"),
    ("query head taken as the kv head", "(size_t)p->num_q_heads + (size_t)h) * (size_t)d;",
     "(size_t)p->num_q_heads + (size_t)g) * (size_t)d;"),
    ("e4m3 zero loses its sign", "const uint8_t sign = signbit(x) ? 0x80 : 0x00;",
     "const uint8_t sign = x < 0 ? 0x80 : 0x00;"),
    ("fp8 write ignores the K scale", "quotient_f32((float)bf16_bits_to_double(key[src + e]), k_scale)",
     "quotient_f32((float)bf16_bits_to_double(key[src + e]), 1.0f)"),
    ("fp8 V read with the K scale", "(which ? p->v_scale : p->k_scale)", "(which ? p->k_scale : p->k_scale)"),
    ("layout heads and k/v swapped", "idx = idx * (size_t)num_kv_heads + (size_t)kv_head;\n    idx = idx * 2u + (size_t)which;",
     "idx = idx * 2u + (size_t)which;\n    idx = idx * (size_t)num_kv_heads + (size_t)kv_head;"),
]

BATTERY = r"""
import sys
sys.path.insert(0, {tests!r}); sys.path.insert(0, {root!r})
import oracle, test_oracle_pins as pins, test_oracle_fp8_pins as f8
tests = [f8.test_decode_matches_torch_on_all_codes,
         f8.test_encode_matches_torch_rounding_inside_its_range,
         f8.test_saturation_and_signed_zero,
         lambda: f8.test_fp8_write_matches_torch_quotient_rounding(0.0173, 3.7),
         lambda: f8.test_fp8_attention_matches_torch_sdpa_on_contiguous_dequantised_kv(0.0173, 3.7),
lambda: [pins.test_oracle_matches_torch_sdpa_on_contiguous_kv(c) for c in range(len(pins.CASES))],
         pins.test_oracle_matches_sdpa_with_shared_prefix_and_forks,
         pins.test_index_example_from_the_pages,
         pins.test_single_key_returns_its_value_exactly,
         pins.test_two_keys_closed_form,
         pins.test_uniform_keys_and_zero_scale_give_the_mean_of_values,
         pins.test_split_key_range_merges_to_the_full_row,
         pins.test_kv_write_round_trip_and_untouched_slots,
         pins.test_copy_on_write_copy_gives_the_fork_the_parents_view]
caught = 0
with oracle.use_library({so!r}):
    for t in tests:
        try:
            t()
        except (AssertionError, oracle.OracleError):
            caught += 1
sys.exit(3 if caught else 0)
"""


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("mutant", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(mutant, source, tmp_path):
    name, old, new = mutant
    assert source.count(old) == 1, f"mutation site for {name!r} not found exactly once"
    c_file = tmp_path / "mutant.c"
    c_file.write_text(source.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(c_file), "-lm"],
                   check=True, capture_output=True)
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = BATTERY.format(tests=tests_dir, root=os.path.dirname(tests_dir), so=str(so))
    # a mutant may also read outside its arrays and crash: any non-zero exit
    # of the battery's own process means the mistake was caught
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"no pin caught the planted mistake {name!r}"


def test_battery_passes_on_the_unmodified_oracle(source, tmp_path):
    c_file = tmp_path / "same.c"
    c_file.write_text(source)
    so = tmp_path / "libsame.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(c_file), "-lm"],
                   check=True, capture_output=True)
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = BATTERY.format(tests=tests_dir, root=os.path.dirname(tests_dir), so=str(so))
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]

"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is a one-expression edit of ``oracle/pkv_oracle.c`` compiled
into a temporary library; the committed oracle is never modified.  For each
one, at least one of the pin tests in ``test_oracle_pins`` must fail.
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
    ("keys read from the V half", "const uint16_t *k = p->cache + cache_offset(phys, g, 0,",
     "const uint16_t *k = p->cache + cache_offset(phys, g, 1,"),
    ("table indexed by offset", "const int32_t phys = table[j / B];\n        const uint16_t *k",
     "const int32_t phys = table[j % B];\n        const uint16_t *k"),
    ("offset taken as block index", "cache_offset(phys, g, 1, (int32_t)(j % B),",
     "cache_offset(phys, g, 1, (int32_t)((j / B) % B),"),
    ("scale dropped", "const double s = p->scale * dot;", "const double s = dot;"),
    ("no normalisation", "        out[e] /= z;\n    *lse = m + log(z);", "        out[e] /= 1.0;\n    *lse = m + log(z);"),
    ("lse without the maximum", "*lse = m + log(z);\n    if (weights)", "*lse = log(z);\n    if (weights)"),
    ("cache write offset", "const int32_t off = (int32_t)(slot % block_size);",
     "const int32_t off = (int32_t)((slot + 1) % block_size);"),
    ("cache write K/V swapped", "memcpy(cache + cache_offset(block, h, 0, off, num_kv_heads, block_size, head_size),\n                   key + src",
     "memcpy(cache + cache_offset(block, h, 0, off, num_kv_heads, block_size, head_size),\n                   value + src"),
    ("combine ignores weights", "const double w = exp(part_lse[s] - m);", "const double w = 1.0;"),
    ("block copy covers one kv head", "const size_t block_elems = cache_offset(1, 0, 0, 0, num_kv_heads, block_size, head_size);",
     "const size_t block_elems = cache_offset(0, 1, 0, 0, num_kv_heads, block_size, head_size);"),
    ("layout heads and k/v swapped", "idx = idx * (size_t)num_kv_heads + (size_t)kv_head;\n    idx = idx * 2u + (size_t)which;",
     "idx = idx * 2u + (size_t)which;\n    idx = idx * (size_t)num_kv_heads + (size_t)kv_head;"),
]

BATTERY = r"""
import sys
sys.path.insert(0, {tests!r}); sys.path.insert(0, {root!r})
import oracle, test_oracle_pins as pins
tests = [lambda: [pins.test_oracle_matches_torch_sdpa_on_contiguous_kv(c) for c in range(len(pins.CASES))],
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

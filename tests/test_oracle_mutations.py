"""Each plausible mistake planted in a copy of the oracle's C source (on the
CPU, in a temporary build) must make at least one pin fail.  This shows the
pins are sharp enough to catch a dropped term, a swapped operand or a wrong
index in the oracle."""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

# (name, text in pa_oracle.c, planted replacement, occurrence to replace)
MUTATIONS = [
    ("dropped scale", "x[j - j0] = scale * dot;", "x[j - j0] = dot;"),
    ("value read from the key plane",
     "double vd = read_elem(cache, cache_index(1,", "double vd = read_elem(cache, cache_index(0,"),
    ("query head mapped modulo", "int h = hq / group;", "int h = hq % num_kv_heads;"),
    ("table indexed by offset", "int64_t b = row[j / block_size];",
     "int64_t b = row[j % block_size];"),
    ("softmax not normalised", "for (int d = 0; d < head_size; ++d) o[d] /= den;",
     "for (int d = 0; d < head_size; ++d) o[d] /= 1.0;"),
    ("new token left out", "int64_t len = seq_lens[s];", "int64_t len = seq_lens[s] - 1;"),
    ("slot split by pool size", "int64_t b = slot / block_size;",
     "int64_t b = slot % num_blocks;"),
    ("copy of keys only", "for (int kv = 0; kv < 2; ++kv) {", "for (int kv = 0; kv < 1; ++kv) {"),
    ("partials combined without their sums", "den += w * part_l[base + p];",
     "den += part_l[base + p];"),
]

PIN_CALLS = [
    lambda: [pins.test_decode_equals_contiguous_sdpa(m) for m in pins.CASES],
    pins.test_decode_gqa_equals_repeated_kv_heads,
    pins.test_reshape_and_cache_places_worked_example_token,
    pins.test_reshape_and_cache_skips_padding_and_matches_numpy_assignment,
    pins.test_copy_blocks_matches_numpy_assignment,
    lambda: pins.test_split_partials_combine_to_single_pass(12),
    pins.test_worked_example_decode_steps_match_contiguous_attention,
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    text = open(SRC).read()
    assert old in text, "mutation site vanished: %s" % name
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new, 1))
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    str(src), "-o", str(so), "-lm"], check=True, capture_output=True)
    saved = oracle._load()
    oracle._lib = oracle.bind(str(so))
    caught = []
    try:
        for call in PIN_CALLS:
            try:
                call()
            except (AssertionError, IndexError):
                caught.append(call)
    finally:
        oracle._lib = saved
    assert caught, "no pin caught the planted mistake '%s'" % name

"""The oracle's pins must be able to fail: plant one plausible mistake at a time in a copy
of the oracle's C source (on the CPU), rebuild it, and check that at least one pin
rejects it.  Nothing here touches the CUDA path."""
import os

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "pagedkv_oracle.c")

GQA_LOOP = "for (int32_t h = g * group; h < (g + 1) * group; ++h) {"

MUTATIONS = {
    "dropped_scale": ("scores[j] = scale * dot;", "scores[j] = dot;",
                      [lambda: pins.test_decode_matches_sdpa(0)]),
    "interleaved_gqa": (GQA_LOOP, "for (int32_t h = g; h < num_q_heads; h += num_kv_heads) {",
                        [lambda: pins.test_decode_matches_sdpa(1), pins.test_gqa_mapping_golden]),
    "causal_off_by_one": ("int32_t visible = L - q_len + i + 1;",
                          "int32_t visible = L - q_len + i;",
                          [lambda: pins.test_prefill_matches_sdpa_causal_square(10)]),
    "chunk_at_start": ("int32_t visible = L - q_len + i + 1;", "int32_t visible = i + 1;",
                       [lambda: pins.test_prefill_matches_sdpa_causal_square(11)]),
    "decode_drops_newest_key": (
        "attend_one_query(q + row * head_dim, K, V, L, head_dim",
        "attend_one_query(q + row * head_dim, K, V, L - 1, head_dim",
        [lambda: pins.test_decode_matches_sdpa(2), pins.test_context_of_one_returns_v_exactly]),
    "slot_transposed": ("(int64_t)phys * block_size + offset", "(int64_t)offset * num_blocks + phys",
                        [pins.test_block_table_worked_example]),
    "pool_head_offset_swapped": (
        "((block * num_kv_heads + head) * block_size + offset) * head_dim + dim",
        "((block * block_size + offset) * num_kv_heads + head) * head_dim + dim",
        [pins.test_scatter_layout_matches_numpy_indexing]),
    "not_normalised": ("double p = scores[j] / l;", "double p = scores[j];",
                       [lambda: pins.test_decode_matches_sdpa(3)]),
    "values_read_from_keys": ("out[d] += p * V[", "out[d] += p * K[",
                              [lambda: pins.test_decode_matches_sdpa(0)]),
    "one_block_too_many": ("while (capacity < tokens)", "while (capacity <= tokens)",
                           [pins.test_block_arithmetic_golden]),
    "value_store_from_key": ("value_cache[dst] = value[src];", "value_cache[dst] = key[src];",
                             [pins.test_scatter_layout_matches_numpy_indexing]),
    "copy_blocks_keys_only": ("          value_cache[to] = value_cache[from];", "",
                              [pins.test_copy_blocks_copies_whole_blocks_in_order]),
    "score_sign_flipped": ("scores[j] = scale * dot;", "scores[j] = -scale * dot;",
                           [pins.test_two_keys_logistic_closed_form]),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new, checks = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = tmp_path / "mutated.c"
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutated), str(tmp_path / "libmutated.so"))
    with oracle.use_library(lib):
        for check in checks:
            with pytest.raises(AssertionError):
                check()

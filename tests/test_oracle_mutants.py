"""Plant plausible mistakes in copies of the oracle source and check that
every one of them fails at least one pin. CPU only."""
import os

import pytest

import oracle

import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement); every mutant stays in bounds
MUTANTS = [
    ("kv_head_modulo", "const int kvh = h / group;", "const int kvh = h % num_kv_heads;"),
    ("head_major_layout", "((block * block_size + t % block_size) * num_kv_heads + kvh)",
     "((block * num_kv_heads + kvh) * block_size + t % block_size)"),
    ("rows_reversed", "(block * block_size + t % block_size)",
     "(block * block_size + (block_size - 1 - t % block_size))"),
    ("scale_dropped", "score[t] = scale * dot;", "score[t] = dot;"),
    ("not_normalised", "double p = score[t] / denom;", "double p = score[t];"),
    ("last_token_dropped", "t < L;", "t < L - 1;"),
    ("query_row_of_kv_head", "(int64_t)q_index * num_q_heads + h) * head_dim",
     "(int64_t)q_index * num_q_heads + kvh) * head_dim"),
    ("causal_diagonal_dropped", "const int cap = context_lens[s] - q_len + i + 1;",
     "const int cap = context_lens[s] - q_len + i;"),
    ("causal_mask_ignored", "const int cap = context_lens[s] - q_len + i + 1;",
     "const int cap = context_lens[s];"),
    ("store_v_from_k", "memcpy(v_cache + slot * row, v + i * row",
     "memcpy(v_cache + slot * row, k + i * row"),
    ("head_major_rows_token_major",
     "? k_cache + ((block * num_kv_heads + kvh) * block_size + t % block_size) * (int64_t)head_dim",
     "? k_cache + ((block * block_size + t % block_size) * num_kv_heads + kvh) * (int64_t)head_dim"),
    ("head_major_store_head_stride", "const int64_t dst = ((block * num_kv_heads + h) * block_size + off) * head_dim;",
     "const int64_t dst = ((block * block_size + off) * num_kv_heads + h) * head_dim;"),
    ("prefill_row_offset", "const int cap = context_lens[s] - n + i + 1;",
     "const int cap = context_lens[s] - n + i;"),
    ("store_skips_first_row", "if (slot == -1)\n            continue;",
     "if (slot == -1 || i == 0)\n            continue;"),
    ("pv_reads_keys",
     ": v_cache + ((block * block_size + t % block_size) * num_kv_heads + kvh) * (int64_t)head_dim;",
     ": k_cache + ((block * block_size + t % block_size) * num_kv_heads + kvh) * (int64_t)head_dim;"),
    ("softmax_base_two", "score[t] = exp(score[t] - mx);", "score[t] = exp2(score[t] - mx);"),
    ("prefill_row_offset_in_batch", "const int i = row - query_start_loc[s];",
     "const int i = row;"),
    ("prefill_boundary_row_to_previous_sequence", "while (query_start_loc[s + 1] <= row)",
     "while (query_start_loc[s + 1] < row)"),
    # decode_pairs, the oracle of the full-size GPU checks
    ("pairs_length_of_first_sequence", "context_lens[pairs[2 * i]], ORACLE_LAYOUT_TOKEN_MAJOR,",
     "context_lens[0], ORACLE_LAYOUT_TOKEN_MAJOR,"),
    ("pairs_query_of_first_sequence", "num_blocks, pairs[2 * i],\n",
     "num_blocks, 0,\n"),
    ("pairs_outputs_reversed", "context_lens[pairs[2 * i]], ORACLE_LAYOUT_TOKEN_MAJOR,\n                           out + i * head_dim);",
     "context_lens[pairs[2 * i]], ORACLE_LAYOUT_TOKEN_MAJOR,\n                           out + (num_pairs - 1 - i) * head_dim);"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    with open(SRC) as fh:
        text = fh.read()
    assert old in text, f"mutation anchor for {name} not found"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    mutant = oracle.compile_variant(str(src), str(tmp_path / "libmutant.so"))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except (AssertionError, oracle.OracleError) as e:
            failed.append((pin.__name__, str(e)[:80]))
    assert failed, f"mutant {name} passed every pin"

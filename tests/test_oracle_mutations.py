"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one (CPU only; the mutated copies are built in a temp folder)."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "csgmv_oracle.c")

# (name, original text, mutated text, pins expected to catch it)
MUTATIONS = [
    ("h_layout_transposed", "ht[(int64_t)j * r + k] = acc;", "ht[(int64_t)k * c + j] = acc;",
     ["fused_dense"]),
    ("padded_slice_stride", "Aw + ((int64_t)j * r + k) * K", "Aw + ((int64_t)j * R + k) * K",
     ["fused_dense"]),
    ("scaling_dropped", "yt[n] += sigma * acc;", "yt[n] += acc;", ["fused_dense"]),
    ("B_operand_transposed", "oracle_bf16_to_f64(Bw[n * R + k])", "oracle_bf16_to_f64(Bw[k * N + n])",
     ["fused_dense"]),
    ("expand_ignores_slice", "acc += ht[(int64_t)j * r + k] *", "acc += ht[k] *", ["fused_dense"]),
    ("shrink_x_index", "oracle_bf16_to_f64(xt[i]) * oracle_bf16_to_f64(arow[i])",
     "oracle_bf16_to_f64(xt[i]) * oracle_bf16_to_f64(arow[K - 1 - i])", ["fused_dense"]),
    ("sort_ties_reversed", "return x->index < y->index ? -1 : 1;", "return x->index < y->index ? 1 : -1;",
     ["perm_example", "brute"]),
    ("segment_count_off_by_one", "int num_segs = (group_len + chunk - 1) / chunk;",
     "int num_segs = group_len / chunk + 1;", ["segments_example", "brute"]),
    ("chunk_rule_boundary", "if (num_tokens >= 256)", "if (num_tokens > 256)", ["chunk_rule"]),
    ("graph_padding_value", "seg_indptr[k + 1] = s;", "seg_indptr[k + 1] = 0;", ["tiny"]),
    ("embedding_ignores_rank", "for (int k = 0; k < r && k < R; ++k)", "for (int k = 0; k < R; ++k)",
     ["embedding"]),
    ("lm_head_empty_request_breaks_run", "if (pruned_lens[i] == 0) continue;",
     "if (pruned_lens[i] == 0) { run_slot[nruns] = -1; run_len[nruns] = 0; ++nruns; continue; }",
     ["lm_head"]),
    ("lm_head_no_merge", "if (nruns > 0 && run_slot[nruns - 1] == req_adapter[i]) {",
     "if (nruns < 0) {", ["lm_head"]),
    ("expand_uses_max_rank", "for (int k = 0; k < r; ++k)\n                    acc += ht[(int64_t)j * r + k] * oracle_bf16_to_f64(Bw[n * R + k]);",
     "for (int k = 0; k < R; ++k)\n                    acc += ht[(int64_t)j * r + k] * oracle_bf16_to_f64(Bw[n * R + k]);",
     ["fused_dense", "padding"]),
    ("sliced_b_global_column", "Bw[(n - off[j]) * R + k]", "Bw[n * R + k]", ["sliced_dense"]),
    ("sliced_b_slot_stride", "Bs[j] + (int64_t)w * width * R", "Bs[j] + (int64_t)w * N * R", ["sliced_dense"]),
    ("extra_row_off_by_one", "extra[((int64_t)w * num_extra + (id - V)) * R + k]",
     "extra[((int64_t)w * num_extra + (id - V + 1) % num_extra) * R + k]", ["embedding_extra"]),
    ("extra_ignores_rank", "for (int k = 0; k < rr; ++k) {", "for (int k = 0; k < R; ++k) {",
     ["embedding_extra"]),
    ("extra_token_overwrites_base_rows", "if (id < V) continue;", "if (id < 0) continue;", ["extra_token"]),
]

PINS = {
    "fused_dense": lambda: [pins.test_fused_matches_dense_delta(s) for s in range(6)],
    "perm_example": pins.test_permutation_worked_example,
    "segments_example": pins.test_segments_worked_example,
    "brute": lambda: [pins.test_builder_brute_force(s) for s in range(40)],
    "chunk_rule": pins.test_chunk_size_rule_table,
    "tiny": pins.test_tiny_batch_info_hand_derived,
    "embedding": pins.test_embedding_is_column_indexing,
    "rank0": pins.test_rank_zero_and_no_adapter_leave_base_exact,
    "padding": pins.test_padding_is_never_read,
    "lm_head": pins.test_lm_head_batch_info_hand_derived,
    "sliced_dense": lambda: [pins.test_sliced_b_matches_dense_delta(s) for s in range(4)],
    "embedding_extra": pins.test_embedding_extra_is_indexing_of_both_tables,
    "extra_token": pins.test_extra_token_embedding_replaces_only_extra_rows,
}


@pytest.mark.parametrize("name,orig,mut,catchers", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, orig, mut, catchers):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor not unique/found: {orig!r}"
    path = tmp_path / f"oracle_{name}.c"
    path.write_text(src.replace(orig, mut))
    so = tmp_path / f"liboracle_{name}.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(path), "-o", str(so)])
    oracle.use_library(str(so))
    try:
        caught = []
        for pin in catchers:
            try:
                PINS[pin]()
            except AssertionError:
                caught.append(pin)
        assert caught, f"planted mistake {name} passed every pin in {catchers}"
    finally:
        oracle.use_library(None)

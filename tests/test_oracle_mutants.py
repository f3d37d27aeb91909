"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Each mutant is compiled from the oracle's C source with one textual change; the
pins must then fail. This shows the pins constrain every step of the oracle (fp16
decoding, score terms, order, tie-break, expansion, trailing pool, remap, guards,
row context) rather than only re-stating it.
"""

import pytest

import oracle
from _pins import ALL_PINS

MUTANTS = {
    "dropped_head": [("for (int h = 0; h < heads; ++h)", "for (int h = 1; h < heads; ++h)")],
    "transposed_q": [("q_row[h * dim + d]", "q_row[d * heads + h]")],
    "wrong_sign_decode": [("return (float)(sign ? -v : v);", "return (float)(v);")],
    "subnormal_scale": [("ldexp((double)frac, -24)", "ldexp((double)frac, -25)")],
    "ties_to_higher_index": [("return a->j < b->j;", "return a->j > b->j;")],
    "ascending_scores": [("return a->s > b->s;", "return a->s < b->s;")],
    "one_pool_short": [("int32_t n = K < P ? K : P;", "int32_t n = K < P ? K - 1 : P;")],
    "no_trailing_pool": [("for (int64_t t = P * kpool; t < ctx; ++t)",
                          "for (int64_t t = P * kpool; t < P * kpool; ++t)")],
    "remap_offset": [("return (int64_t)ph * block_stride_rows + (t % block_size);",
                      "return (int64_t)ph * block_stride_rows + (t / block_size);")],
    "remap_stride_is_block": [("return (int64_t)ph * block_stride_rows + (t % block_size);",
                               "return (int64_t)ph * block_size + (t % block_size);")],
    "missing_block_guard": [("if (b >= max_blocks)", "if (b > max_blocks)")],
    "missing_physical_guard": [("if (ph < 0 || ph >= num_kv_blocks)", "if (ph < 0)")],
    "context_is_position": [("int64_t ctx = (int64_t)p->positions[r] + 1;",
                             "int64_t ctx = (int64_t)p->positions[r];")],
    "key_row_from_page": [("(int64_t)(j % p->key_page_size) * p->dim",
                           "(int64_t)(j / p->key_page_size) * p->dim"),
                          ("(j % p->key_page_size) * p->dim", "(j / p->key_page_size) * p->dim")],
    "kept_pools_not_sorted": [("    qsort(out, (size_t)n, sizeof(int32_t), orc_cmp_int);\n", "")],
    "workspace_start_ignored": [("s = (int64_t)ws_starts[w] + t;", "s = (int64_t)t;")],
    "workspace_rows_use_global": [("if (w == -1) {", "if (w >= -1) {")],
    "dcp_owner_by_token": [("if (group % dcp_size != dcp_rank)", "if (t % dcp_size != dcp_rank)")],
    "dcp_local_drops_offset": [("return (group / dcp_size) * interleave + t % interleave;",
                                "return (group / dcp_size) * interleave;")],
    "dcp_local_not_divided": [("return (group / dcp_size) * interleave + t % interleave;",
                               "return group * interleave + t % interleave;")],
    "dcp_table_not_dense": [("num_kv_blocks, block_size, block_size);", "num_kv_blocks, block_size, 2 * block_size);")],
    "maxsim_min_not_max": [("                if (s > best)\n", "                if (s < best || best == -INFINITY)\n")],
    "maxsim_max_starts_at_zero": [("double best = -INFINITY, best_abs = 0.0;", "double best = 0.0, best_abs = 0.0;")],
    "maxsim_last_row_dropped": [("for (int32_t j = 0; j < lengths[i]; ++j) {", "for (int32_t j = 0; j < lengths[i] - 1; ++j) {")],
    "maxsim_q_transposed": [("orc_half_to_float(q[(int64_t)a * d + k])", "orc_half_to_float(q[(int64_t)k * lq + a])")],
    "maxsim_stride_is_d": [("const uint16_t *row = docs + r * doc_stride;", "const uint16_t *row = docs + r * d;")],
    "maxsim_first_query_row_only": [("for (int32_t a = 0; a < lq; ++a) {\n            double best", "for (int32_t a = 0; a < 1; ++a) {\n            double best")],
    "maxsim_oob_not_zero": [("double s = 0.0, sa = 0.0;\n                if (r >= 0", "double s = -1.0, sa = 0.0;\n                if (r >= 0")],
    "bf16_wrong_shift": [("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;")],
    "mla_no_max_shift": [("const double p = exp(logit[j] - m);", "const double p = exp(logit[j]);")],
    "mla_scale_dropped": [("logit[j] = sm_scale * acc;", "logit[j] = acc;")],
    "mla_rope_dropped": [("for (int32_t d = 0; d < dr; ++d)\n                    acc +=",
                          "for (int32_t d = 0; d < 0; ++d)\n                    acc +=")],
    "mla_kv_len_ignored": [("const int32_t n = kv_len[r] < width ? kv_len[r] : width;", "const int32_t n = width;")],
    "mla_not_normalised": [("o[d] /= z;", "o[d] /= 1.0;")],
    "mla_lse_without_max": [("lse[(int64_t)r * heads + h] = m + log(z);", "lse[(int64_t)r * heads + h] = log(z);")],
    "dcp_compact_keeps_columns": [("                    out[cnt] = s;", "                    out[c] = s;")],
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    so = oracle.build_variant(MUTANTS[name], name)
    failed = []
    with oracle.using_library(so):
        for pin in ALL_PINS:
            try:
                pin(oracle)
            except AssertionError:
                failed.append(pin.__name__)
                break
    assert failed, f"no pin caught the planted mistake {name}"

"""Planted mistakes: each test compiles a copy of the oracle with one
plausible error (a wrong index, sign, operand or constant) and checks that
the pins in test_oracle_pins catch it.  Runs on the CPU only.  Every planted
error keeps all memory accesses inside the buffers the pins pass."""
import contextlib
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_bsr_mask as mpins
from tests import test_oracle_fp8 as fpins
from tests import test_oracle_pins as pins
from tests import test_oracle_softcap as cpins
from tests import test_oracle_varbsr as vpins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sfa_oracle.c")

# (name, original text, planted text)
MUTANTS = [
    ("gqa_head_map", "const int n2 = n1 / G;", "const int n2 = n1 % s->N2;"),
    ("causal_off_by_one", "if (s->causal && id > diag)", "if (s->causal && id >= diag)"),
    ("causal_top_left", "const int diag = s1 + (s->S2 - s->S1);", "const int diag = s1;"),
    ("scale_dropped", "scores[i] = dot * s->scale;", "scores[i] = dot;"),
    ("softmax_unnormalised", "weights[i] /= sum;", "weights[i] /= 1.0;"),
    ("lse_base2", "weights[i] /= sum;\n    if (lse_row) *lse_row = mx + log(sum);",
     "weights[i] /= sum;\n    if (lse_row) *lse_row = mx + log2(sum);"),
    ("bsr_lse_base2", "y_row[e] += w * (sv * oracle_elem(v, vo + e, s->kv_dtype));\n    }\n    if (lse_row) *lse_row = mx + log(sum);",
     "y_row[e] += w * (sv * oracle_elem(v, vo + e, s->kv_dtype));\n    }\n    if (lse_row) *lse_row = mx + log2(sum);"),
    ("varbsr_lse_base2", "* d + e, s->dtype);\n    }\n    if (lse_row) *lse_row = mx + log(sum);",
     "* d + e, s->dtype);\n    }\n    if (lse_row) *lse_row = mx + log2(sum);"),
    ("bnsd_index_as_bsnd", ": (((int64_t)b * s->N2 + n2) * s->S1 + s1) * s->topK;",
     ": (((int64_t)b * s->S1 + s1) * s->N2 + n2) * s->topK;"),
    ("value_stride_dv", "const int64_t vo = row_kv(s, b, n2, si[i]) * s->ldv;",
     "const int64_t vo = row_kv(s, b, n2, si[i]) * s->Dv;"),
    ("value_row_from_slot", "const int64_t vo = row_kv(s, b, n2, si[i]) * s->ldv;",
     "const int64_t vo = row_kv(s, b, n2, i) * s->ldv;"),
    ("masked_row_not_zero", "for (int e = 0; e < s->Dv; ++e) y_row[e] = 0.0;\n        if (lse_row) *lse_row = -INFINITY;",
     "for (int e = 0; e < s->Dv; ++e) y_row[e] = 1.0;\n        if (lse_row) *lse_row = -INFINITY;"),
    ("bsr_kv_head_map", "const int kvh = h / (s->Hq / s->Hkv);", "const int kvh = h % s->Hkv;"),
    ("bsr_block_col_unscaled", "allowed[(int64_t)indices[jj] * s->C + c] = ok;",
     "allowed[(int64_t)indices[jj] + c] = ok;"),
    ("bsr_mask_bit_order_lsb", "(s->packed_mask[e >> 3] >> (7 - (e & 7))) & 1",
     "(s->packed_mask[e >> 3] >> (e & 7)) & 1"),
    ("bsr_mask_row_in_block", "((int64_t)jj * s->R + (i - br * s->R)) * s->C + c",
     "((int64_t)jj * s->R) * s->C + c"),
    ("bsr_causal_top_left", "if ((int64_t)j > (int64_t)i + (s->N - s->M)) allowed[j] = 0;",
     "if ((int64_t)j > (int64_t)i) allowed[j] = 0;"),
    ("bsr_causal_with_mask", "if (!s->packed_mask && s->causal)", "if (s->causal)"),
    ("bsr_row_block_reversed", "const int br = i / s->R;", "const int br = (s->M - 1 - i) / s->R;"),
    ("bsr_scale_dropped", "(sk * oracle_elem(k, ko + e, s->kv_dtype));\n        scores[j] = oracle_soft_cap(dot * s->scale,",
     "(sk * oracle_elem(k, ko + e, s->kv_dtype));\n        scores[j] = oracle_soft_cap(dot,"),
    ("varbsr_scale_dropped", "* d + e, s->dtype);\n        scores[j] = oracle_soft_cap(dot * s->scale,",
     "* d + e, s->dtype);\n        scores[j] = oracle_soft_cap(dot,"),
    ("varbsr_kv_head_map", "i = (int)(r % s->M), g = h / G;", "i = (int)(r % s->M), g = h % s->Hkv;"),
    ("varbsr_row_block_off_by_one", "while (acc + row_sz[(int64_t)g * MB + rb] <= i)",
     "while (acc + row_sz[(int64_t)g * MB + rb] < i)"),
    ("varbsr_col_sizes_of_head0", "for (int c = 0; c < col_sz[(int64_t)g * NB + cb]; ++c)",
     "for (int c = 0; c < col_sz[cb]; ++c)"),
    ("varbsr_mask_map_transposed", "mask_map[((int64_t)g * MB + rb) * NB + colblk[j]]",
     "mask_map[((int64_t)g * NB + colblk[j]) * MB + rb]"),
    ("varbsr_causal_top_left", "if (s->causal && (int64_t)j > (int64_t)i + (N - M)) allowed[j] = 0;",
     "if (s->causal && (int64_t)j > (int64_t)i) allowed[j] = 0;"),
    ("softcap_before_scale", "* d + e, s->dtype);\n        scores[j] = oracle_soft_cap(dot * s->scale, s->softcap);",
     "* d + e, s->dtype);\n        scores[j] = oracle_soft_cap(dot, s->softcap) * s->scale;"),
    ("softcap_no_multiplier", "return cap > 0.0 ? cap * tanh(x / cap) : x;",
     "return cap > 0.0 ? tanh(x / cap) : x;"),
    ("softcap_ignored_in_bsr", "(sk * oracle_elem(k, ko + e, s->kv_dtype));\n        scores[j] = oracle_soft_cap(dot * s->scale, s->softcap);",
     "(sk * oracle_elem(k, ko + e, s->kv_dtype));\n        scores[j] = dot * s->scale;"),
    ("bf16_as_f16", "return dtype == 1 ? oracle_bf16(p[i]) : oracle_f16(p[i]);",
     "return oracle_f16(p[i]);"),
    # FP8 formats and per-head scales
    ("e4m3_exponent_bias", "else v = ldexp((double)(8 + m), e - 10);",
     "else v = ldexp((double)(8 + m), e - 11);"),
    ("e4m3_subnormal_as_normal", "if (e == 0) v = ldexp((double)m, -9);",
     "if (e == 0) v = ldexp((double)(8 + m), -10);"),
    ("e4m3_no_nan", "if (e == 15 && m == 7) return NAN;", "if (e == 16) return NAN;"),
    ("e5m2_mantissa_width", "else v = ldexp((double)(4 + m), e - 17);",
     "else v = ldexp((double)(8 + m), e - 18);"),
    ("e5m2_read_as_e4m3", "default: return oracle_e5m2(((const uint8_t*)p)[i]);",
     "default: return oracle_e4m3(((const uint8_t*)p)[i]);"),
    ("scale_q_by_kv_head", "const double sq = s->scale_q ? s->scale_q[h] : 1.0;",
     "const double sq = s->scale_q ? s->scale_q[kvh] : 1.0;"),
    ("scale_k_by_qo_head", "const double sk = s->scale_k ? s->scale_k[kvh] : 1.0;",
     "const double sk = s->scale_k ? s->scale_k[h % s->Hkv] : 1.0;"),
    ("scale_v_dropped", "y_row[e] += w * (sv * oracle_elem(v, vo + e, s->kv_dtype));",
     "y_row[e] += w * oracle_elem(v, vo + e, s->kv_dtype);"),
    ("scale_v_as_scale_k", "const double sv = s->scale_v ? s->scale_v[kvh] : 1.0;",
     "const double sv = s->scale_k ? s->scale_k[kvh] : 1.0;"),
    ("q_read_with_kv_type", "dot += (sq * oracle_elem(q, qo + e, s->q_dtype)) *",
     "dot += (sq * oracle_elem(q, qo + e, s->kv_dtype)) *"),
]


def all_pins():
    """Every pin with its parameters, as zero-argument callables."""
    out = []
    for layout in ("BSND", "BNSD"):
        for causal in (False, True):
            for dtype in ("f16", "bf16"):
                out.append(lambda l=layout, c=causal, d=dtype: pins.test_brute_force_multiset(l, c, d))
            out.append(lambda l=layout, c=causal: pins.test_identity_indices_equal_dense_sdpa(l, c))
        out.append(lambda l=layout: pins.test_value_prefix_view_equals_copy(l))
    out += [pins.test_causal_mask_matches_printed_rule, pins.test_fully_masked_rows_are_zero,
            pins.test_single_slot_closed_form, pins.test_uniform_scores_give_mean,
            pins.test_bsr_worked_example, pins.test_bsr_empty_block_row_is_zero]
    for args in ((3, 2, 10, 8), (4, 4, 12, 16), (1, 3, 5, 9)):
        out.append(lambda a=args: pins.test_bsr_equals_block_expanded_mask(*a))
    # block-sparse mask / causal pins
    out += [mpins.test_full_mask_equals_no_mask, mpins.test_mask_overrides_causal,
            mpins.test_packed_bit_order_most_significant_first, mpins.test_fully_masked_rows_zero]
    for mn in ((128, 128), (96, 128)):
        out.append(lambda a=mn: mpins.test_causal_matches_dense_bottom_right(*a))
    out.append(lambda: mpins.test_mask_matches_dense(0.3))
    # variable block-sparse pins
    out += [vpins.test_worked_example_expands_as_printed, vpins.test_kv_heads_keep_their_own_masks,
            vpins.test_single_block_equals_dense_sdpa, vpins.test_empty_blocks_and_fully_masked_rows,
            vpins.test_uniform_keys_give_mean_of_allowed_values]
    for causal in (False, True):
        out.append(lambda c=causal: vpins.test_matches_dense_brute_force(c, "f16"))
    # soft-cap pins
    out += [cpins.test_large_cap_is_no_cap, cpins.test_tiny_cap_gives_mean_of_allowed_values,
            lambda: cpins.test_bsr_matches_dense_brute_force("plain", 0.7),
            lambda: cpins.test_varbsr_matches_dense_brute_force(False)]
    # FP8 decoding and scale pins
    out += [fpins.test_e4m3_decode_matches_torch, fpins.test_e5m2_decode_matches_torch,
            fpins.test_fp8_closed_forms, fpins.test_e5m2_is_the_high_byte_of_f16,
            fpins.test_fp8_equals_the_16bit_run_on_the_same_values,
            fpins.test_scale_v_scales_the_output_only, fpins.test_scale_k_is_a_per_group_sm_scale,
            fpins.test_scale_q_is_a_per_head_sm_scale]
    for kv in ("e4m3", "e5m2"):
        out.append(lambda t=kv: fpins.test_matches_dense_brute_force(t, "f16"))
        out.append(lambda t=kv: fpins.test_matches_dense_brute_force(t, t))
    return out


@contextlib.contextmanager
def mutant_oracle(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path_c = tmp_path / f"{name}.c"
    path_c.write_text(src.replace(old, new))
    path_so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-o", str(path_so),
                           str(path_c), "-lm"])
    saved = oracle._load()
    oracle._lib = oracle.load_library(str(path_so))
    try:
        yield
    finally:
        oracle._lib = saved


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    caught = 0
    with mutant_oracle(tmp_path, name, old, new):
        for pin in all_pins():
            try:
                pin()
            except (AssertionError, oracle.OracleError):
                caught += 1
    assert caught > 0, f"no pin caught the planted mistake '{name}'"

"""Planted mistakes in copies of the oracle: each must fail at least one pin.

Every mutant is the oracle's C source with one plausible slip (a dropped term,
a wrong sign, index or comparison, a swapped operand), compiled on the CPU into
a temporary library and run through the same pins as the real oracle.
"""
import os

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "scale_over_dk": ("1.0 / sqrt((double)d_k)", "1.0 / (double)d_k"),
    "no_scale": ("scale > 0.0 ? scale : 1.0 / sqrt((double)d_k)", "scale > 0.0 ? scale : 1.0"),
    "causal_hides_diagonal": ("!(causal && j > i)", "!(causal && j >= i)"),
    "causal_reversed": ("!(causal && j > i)", "!(causal && j < i)"),
    "padding_off_by_one": ("(j < len) &&", "(j <= len) &&"),
    "no_normalisation": ("double w = scores[j] / l;", "double w = scores[j];"),
    "max_shift_wrong_sign": ("exp(scores[j] - m)", "exp(m - scores[j])"),
    "no_max_shift": ("exp(scores[j] - m)", "exp(scores[j])"),
    "key_is_value": ("const float* kj = k + (int64_t)j * k_stride;",
                     "const float* kj = v + (int64_t)j * v_stride;"),
    "value_column_index": ("out[c] += w * (double)vj[c];", "out[c] += w * (double)vj[0];"),
    "query_row_index": ("const float* q = c->q + flat * c->d_k;", "const float* q = c->q + (flat / c->n_q) * c->n_q * c->d_k;"),
    "length_of_other_batch": ("int len = clamp_len(c->kv_lengths, c->mask_kind, bi, c->n_k);",
                              "int len = clamp_len(c->kv_lengths, c->mask_kind, 0, c->n_k);"),
    "masked_row_not_zero": ("if (!any) return;               /* every key masked: output row is 0 */",
                            "if (!any) { for (int c = 0; c < d_v; ++c) out[c] = v[c]; return; }"),
    "mha_heads_share_query": ("attention_row_f64(qp + hi * c->d_k,", "attention_row_f64(qp,"),
    "mha_concat_reversed": ("concat + hi * c->d_v, hdk, hdv,", "concat + (c->h - 1 - hi) * c->d_v, hdk, hdv,"),
    "mha_value_uses_key_weights": ("proj_ctx pv = {xkv + (int64_t)bi * n_k * d_model, wv, vp, d_model, hdv};",
                                   "proj_ctx pv = {xkv + (int64_t)bi * n_k * d_model, wk, vp, d_model, hdv};"),
    "window_reach_swapped": ("(int64_t)((r - 1) / 2), (int64_t)(r / 2), rows",
                             "(int64_t)(r / 2), (int64_t)((r - 1) / 2), rows"),
    "window_left_exclusive": ("(j >= i - left)", "(j > i - left)"),
    "window_right_exclusive": ("(j <= i + right)", "(j < i + right)"),
    "decode_position_unshifted": ("int pos = len - c->n_q + i;", "int pos = i;"),
    "decode_position_off_by_one": ("int pos = len - c->n_q + i;", "int pos = len - c->n_q + i + 1;"),
    "backward_ds_sign": ("double ds = prow[j] * (dprow[j] - Di);", "double ds = prow[j] * (dprow[j] + Di);"),
    "backward_dk_unscaled": ("dkj[x] += c->scale * ds * (double)qi[x];", "dkj[x] += ds * (double)qi[x];"),
    "backward_dv_uses_dp": ("dvj[x] += prow[j] * (double)doi[x];", "dvj[x] += dprow[j] * (double)doi[x];"),
    "backward_given_output_no_head_offset": (
        "const float* oi = c->out + bh * (int64_t)c->n_q * c->d_v + (int64_t)i * c->d_v;",
        "const float* oi = c->out + (int64_t)i * c->d_v;"),
    "backward_given_output_not_reset": ("        Di = 0.0;\n        for (int x = 0; x < c->d_v; ++x) Di +=",
                                        "        for (int x = 0; x < c->d_v; ++x) Di +="),
    "backward_given_output_squared": ("Di += (double)doi[x] * (double)oi[x];",
                                      "Di += (double)oi[x] * (double)oi[x];"),
    "lse_drops_max": ("c->lse[r] = m + log(l);", "c->lse[r] = log(l);"),
    "lse_log2": ("c->lse[r] = m + log(l);", "c->lse[r] = m + log2(l);"),
    "lse_unscaled": ("s[j] = c->scale * dot;", "s[j] = dot;"),
    "lse_causal_reversed": ("int visible = (j < len) && !(causal && j > i) && (j >= i - c->left)",
                            "int visible = (j < len) && !(causal && j < i) && (j >= i - c->left)"),
    "mha_output_skips_wo": ("yr[o] += concat[t] * (double)wt[o];", "yr[o] += (o == t) ? concat[t] : 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation site not found: %r" % old
    mutated = tmp_path / ("oracle_%s.c" % name)
    mutated.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutated), str(tmp_path / ("lib_%s.so" % name)))
    o = oracle.Oracle(lib)
    failed = []
    for pin in PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, "mutant %s passed every pin" % name

"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is the oracle's C source with one textual change (a dropped
term, a wrong index or sign, a transposed operand, an off-by-one), compiled
into a temporary library.  The real oracle source is never modified.  A pin
set that lets a mutant through is too weak to trust the oracle.
"""
import importlib.util
import os

import pytest

from tests.oracle_pins import ALL_PINS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

MUTANTS = {
    "gqa_interleaved_mapping": ("int kvh = h / g;", "int kvh = h % Hkv;"),
    "scale_dropped": ("x[t - t0] = scale * acc;", "x[t - t0] = acc;"),
    "max_not_subtracted": ("double p = exp(x[t - t0] - m);", "double p = exp(x[t - t0]);"),
    "row_in_block_off_by_one": ("cache_off(b, t % bs, kvh, 0, bs, Hkv, d);\n        double acc",
                                "cache_off(b, (t + 1) % bs, kvh, 0, bs, Hkv, d);\n        double acc"),
    "cache_axes_transposed": ("return ((b * bs + o) * (int64_t)Hkv + kvh) * d + i;",
                              "return ((b * Hkv + kvh) * (int64_t)bs + o) * d + i;"),
    "output_not_normalised": ("        o[i] /= l;\n    *m_out", "        o[i] /= 1.0;\n    *m_out"),
    "merge_weight_drops_exp_sum": ("double w = exp(max_logits[u * NP + p] - M) * exp_sums[u * NP + p];",
                                   "double w = exp(max_logits[u * NP + p] - M);"),
    "merge_sign_flipped": ("double w = exp(max_logits[u * NP + p] - M)",
                           "double w = exp(M - max_logits[u * NP + p])"),
    "partition_end_off_by_one": ("int t1 = (t0 + P < L) ? t0 + P : L;",
                                 "int t1 = (t0 + P < L) ? t0 + P - 1 : L;"),
    "partition_count_floor": ("        int n = (int)((L + (int64_t)P - 1) / P);\n        int kvh",
                              "        int n = (int)(L / P);\n        int kvh"),
    "bf16_decode_shift": ("((uint32_t)h) << 16;", "((uint32_t)h) << 15;"),
    "f16_subnormal_exponent": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "block_index_uses_modulo": ("int64_t b = bt[(int64_t)s * max_blocks + t / bs];",
                                "int64_t b = bt[(int64_t)s * max_blocks + t % bs];"),
    "query_head_not_used": ("q + ((int64_t)s * Hq + h) * d", "q + ((int64_t)s * Hq + 0) * d"),
    "prefill_causal_off_by_one": ("int p = L - n + (int)(r - q_start[s]);",
                                  "int p = L - n + (int)(r - q_start[s]) + 1;"),
    "prefill_prefix_ignored": ("int p = L - n + (int)(r - q_start[s]);",
                               "int p = (int)(r - q_start[s]);"),
    "prefill_wrong_query_row": ("q + (r * Hq + h) * d", "q + ((int64_t)s * Hq + h) * d"),
    "topk_tie_goes_to_higher_index": ("(best < 0 || x[e] > x[best])",
                                      "(best < 0 || x[e] >= x[best])"),
    "topk_max_not_subtracted": ("if (x[e] > m)\n                m = x[e];",
                                "if (x[e] > m)\n                m = 0.0;"),
    "topk_renormalize_skipped": ("weights[(int64_t)t * k + j] /= sel;",
                                 "weights[(int64_t)t * k + j] /= 1.0;"),
    "sort_not_stable": ("for (int p = 0; p < P; ++p)\n            if (expert_ids[p] == e)",
                        "for (int p = P - 1; p >= 0; --p)\n            if (expert_ids[p] == e)"),
    "sort_offset_off_by_one": ("offsets[e] = r;", "offsets[e] = r + 1;"),
    "gather_pair_index_as_token": ("int t = sorted_pairs[r] / K;", "int t = sorted_pairs[r] % K;"),
    "scatter_weight_dropped": ("o[i] += w * oracle_half_bits_to_f64(row[i], dtype);",
                               "o[i] += oracle_half_bits_to_f64(row[i], dtype);"),
    "scatter_pair_index_not_position": ("int r = pair_pos[(int64_t)t * K + k];",
                                        "int r = (int)((int64_t)t * K + k);"),
}


def _mutant_oracle(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation {name} does not apply"
    mdir = tmp_path / name
    mdir.mkdir()
    (mdir / "pa_oracle.c").write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{name}",
                                                  os.path.join(ROOT, "oracle", "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(mdir / "pa_oracle.c")
    mod._BUILD_DIR = str(mdir / "_build")
    mod._LIB_PATH = str(mdir / "_build" / "libpa_oracle.so")
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    mod = _mutant_oracle(tmp_path, name, old, new)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # AssertionError, or a rejected input
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin detects mutant {name}"

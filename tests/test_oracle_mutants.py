"""The pins must catch plausible mistakes in the oracle.

Each case copies oracle.c to a temporary directory, plants one mistake (a
dropped term, a wrong sign or index, a swapped operand, an off-by-one in the
acceptance rule), builds it, and runs the pin battery of test_oracle_pins.py
against that build: at least one pin has to fail. The mistakes live only in
the temporary copy, on the CPU.
"""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "drop_attention_residual": (
        "t->x[i] = orc_bf16(orc_f32(t->x[i]) + orc_f32(t->att[i]));", "t->x[i] = t->att[i];"),
    "rope_sign": ("float lo = a * c - b * s;", "float lo = a * c + b * s;"),
    "rope_pair_partner": ("float a = orc_f32(x[i]), b = orc_f32(x[i + half]);",
                          "float a = orc_f32(x[i]), b = orc_f32(x[(i + half + 1) % d]);"),
    "gqa_head_map": ("int kvh = h / group;", "int kvh = h % Hkv;"),
    "context_off_by_one": ("pos + 1,\n               d, stride", "pos,\n               d, stride"),
    "no_score_scale": ("s[j] = dot * scale;", "s[j] = dot;"),
    "gate_up_swapped": ("orc_glu(t->gu, t->gu + F, F, c->act, t->a);",
                        "orc_glu(t->gu + F, t->gu, F, c->act, t->a);"),
    # the two intermediate bf16 roundings of the stated rounding path
    "rmsnorm_intermediate_round_dropped": (
        "y[i] = orc_bf16(rb(orc_f32(x[i]) * rstd) * orc_f32(g[i]));",
        "y[i] = orc_bf16(orc_f32(x[i]) * rstd * orc_f32(g[i]));"),
    "glu_activation_round_dropped": ("a[i] = orc_bf16(rb(y) * u);", "a[i] = orc_bf16(y * u);"),
    "layer_entry_cache_offset": ("layer_rest(c, w, layer, pos + r, &t, kb, vb);",
                                 "layer_rest(c, w, layer, pos + r, &t, kb + row, vb + row);"),
    "norm_gain_dropped": ("y[i] = orc_bf16(rb(orc_f32(x[i]) * rstd) * orc_f32(g[i]));",
                          "y[i] = orc_bf16(rb(orc_f32(x[i]) * rstd));"),
    "accept_compares_wrong_row": ("while (n < K - 1 && tokens[n + 1] == am[n]) ++n;",
                                  "while (n < K - 1 && tokens[n] == am[n]) ++n;"),
    "truncate_drops_pending_row": ("m->len = len0 + 1 + n;", "m->len = len0 + n;"),
    "argmax_tie_to_highest": ("if (v[i] > v[best]) best = i;", "if (v[i] >= v[best]) best = i;"),
    "rmsnorm_mean_over_wrong_n": ("ss / (float)n + eps", "ss / (float)(n - 1) + eps"),
    "linear_row_stride": ("const uint16_t* w = W + (size_t)r * cols;",
                          "const uint16_t* w = W + (size_t)r * (cols - 1);"),
}

BATTERY = [
    lambda: pins.test_model_matches_float64_library_decoder(0.1, 0, 1),
    lambda: pins.test_model_matches_float64_library_decoder(0.1, 1, 0),
    lambda: pins.test_rmsnorm_constant_vector(),
    lambda: pins.test_rmsnorm_rounding_points_match_library_casts(),
    lambda: pins.test_glu_rounding_points_match_library_casts(0),
    lambda: pins.test_glu_rounding_points_match_library_casts(1),
    lambda: pins.test_linear_matches_matmul(),
    lambda: pins.test_rope_basis_vectors(64, 1e4),
    lambda: pins.test_rope_depends_on_relative_position_only(),
    lambda: pins.test_attention_single_position_returns_value(),
    lambda: pins.test_attention_matches_sdpa(),
    lambda: pins.test_gqa_head_mapping_matters(),
    *[(lambda r=r: pins.test_argmax_matches_page_selection(r))
      for r in pins._rows("p3_position60_table.txt")],
    lambda: pins.test_verify_rows_equal_decode_and_accept_longest_prefix(_tiny()),
    lambda: pins.test_truncate_then_continue_equals_fresh(_tiny()),
    lambda: pins.test_layer_entry_chain_equals_verify(_tiny()),
]

_TINY = None


def _tiny():
    global _TINY
    if _TINY is None:
        import inputs
        _TINY = (inputs.TINY, inputs.host_weights(inputs.TINY, seed=0, gain_std=0.1))
    return _TINY


def _build_mutant(tmp_path, old, new):
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    d = tmp_path / "mut"
    d.mkdir()
    shutil.copy(os.path.join(ROOT, "oracle", "oracle.h"), d / "oracle.h")
    (d / "oracle.c").write_text(src.replace(old, new))
    so = d / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-o",
                    str(so), str(d / "oracle.c"), "-lm"], check=True)
    return str(so)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    so = _build_mutant(tmp_path, old, new)
    caught = []
    with oracle.use_library(so):
        for i, check in enumerate(BATTERY):
            try:
                check()
            except (AssertionError, ValueError, FloatingPointError):
                caught.append(i)
                break
    assert caught, f"no pin failed for the planted mistake {name!r}"


def test_unmutated_copy_passes_battery(tmp_path):
    so = _build_mutant(tmp_path, "int32_t best = 0;", "int32_t best = 0;")
    with oracle.use_library(so):
        for check in BATTERY:
            check()

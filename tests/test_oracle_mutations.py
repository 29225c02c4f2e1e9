"""Plants plausible mistakes in a copy of the oracle (on the CPU) and checks that the pin
suite rejects every one of them: evidence that the pins constrain each part of it."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTATIONS = {
    "interleaved_group_mapping": ("return h / group;", "return h % p->Nkv;"),
    "causal_off_by_one": ("ORC_CAUSAL_NONE && j > pos)", "ORC_CAUSAL_NONE && j >= pos)"),
    "window_off_by_one": ("j < pos - p->window + 1)", "j < pos - p->window)"),
    "dropped_scale": ("const double raw = p->scale * dot;", "const double raw = dot;"),
    "sink_left_out_of_denominator": ("double l = has_sink ? exp(sink - m) : 0.0;", "double l = 0.0;"),
    "nonpad_off_by_one": ("ORC_LEN_NONPAD_I64 && j >= len_of(p, b))", "ORC_LEN_NONPAD_I64 && j > len_of(p, b))"),
    "mask_sign": (": capped(p, raw + addv) + filt;", ": capped(p, raw - addv) + filt;"),
    "q_bias_segment_ignores_head": ("p->q_bias, h * p->H + d)", "p->q_bias, d)"),
    "filter_as_exclusion": ("ORC_LEN_KEYLEN_I32 && j >= len_of(p, b)) filt += p->mask_filter_value;",
                            "ORC_LEN_KEYLEN_I32 && j >= len_of(p, b)) excluded = 1;"),
    "softcap_missing_outer_factor": ("return p->softcap * tanh(x / p->softcap);", "return tanh(x / p->softcap);"),
    "qk_mode0_includes_bias": ("out[j] = w->raw[j]; return;", "out[j] = w->nocap[j]; return;"),
    "qk_mode1_keeps_excluded_scores": ("w->nocap[j] = excluded ? -INFINITY : nocap;", "w->nocap[j] = nocap;"),
    "qk_mode2_before_softcap": ("out[j] = w->s[j]; return;", "out[j] = w->nocap[j]; return;"),
    "qk_mode3_unnormalised": ("exp(w->s[j] - m) / l : 0.0;", "exp(w->s[j] - m) : 0.0;"),
    "bwd_delta_dropped": ("const double ds = prob[j] * (dp[j] - delta) * p->scale;",
                          "const double ds = prob[j] * dp[j] * p->scale;"),
    "bwd_scale_dropped": ("const double ds = prob[j] * (dp[j] - delta) * p->scale;",
                          "const double ds = prob[j] * (dp[j] - delta);"),
    "bwd_dk_from_probabilities": ("dkr[d] += ds * w.q[d];", "dkr[d] += prob[j] * w.q[d];"),
    "bwd_dv_from_score_gradient": ("dvr[d] += prob[j] * dyrow[d];", "dvr[d] += ds * dyrow[d];"),
    "lower_right_shift": ("pos = valid_total - p->S + i;", "pos = valid_total - p->S + i + 1;"),
    "f16_exponent_bias": ("e - 25);", "e - 24);"),
    "past_not_first": ("if (j < p->P) {", "if (j >= p->L) {"),
    "kv_bias_on_values_uses_key_width": ("kh * D + d)", "kh * p->H + d)"),
    "rotary_sign": ("o[i1] = x1 * c - x2 * sn;", "o[i1] = x1 * c + x2 * sn;"),
    "rotary_pairs_adjacent_always": ("const int64_t i2 = interleaved ? 2 * d + 1 : d + half;",
                                     "const int64_t i2 = 2 * d + 1;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    lib = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                           str(mutated), "-o", str(lib), "-lm"])
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch the planted mistake {name}"

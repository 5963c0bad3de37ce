"""The oracle's pins are strong enough to catch plausible mistakes: each case
below plants one mistake in a copy of the oracle's C source (nibble order,
scale, rounding, sign of the bias, router bias or K range, tie-break,
renormalisation, SwiGLU operand order, stable token order, shared expert,
down projection index, the RMS norm's mean, eps and weight, the residual add
after the layer, the attention's head groups, scale, normalisation and
position range), builds it, and runs the pins against it; at least
one pin must fail.  The shipped oracle is never modified."""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

MUTANTS = [
    ("nibble_order_plain", "return p / 2 + 4 * (p % 2);", "return p;"),
    ("scale_over_16", "float s_exact = range / 15.0f;", "float s_exact = range / 16.0f;"),
    ("code_rounds_down", "float rq = nearbyintf(t);", "float rq = floorf(t);"),
    ("bias_subtracted", "return s * (double)code + b;", "return s * (double)code - b;"),
    ("router_bias_dropped", "acc = acc + router_bias[e];", "acc = acc + 0.0f;"),
    ("router_misses_last_column", "for (int32_t h = 0; h < H; ++h) {\n                float prod",
     "for (int32_t h = 0; h < H - 1; ++h) {\n                float prod"),
    ("ties_to_higher_index", "return (a->expert > b->expert) - (a->expert < b->expert);",
     "return (a->expert < b->expert) - (a->expert > b->expert);"),
    ("weights_not_renormalised",
     "w[j] = renorm ? (exp((double)s[j].logit - mx) / total) / picked : exp((double)s[j].logit - mx) / total;",
     "w[j] = exp((double)s[j].logit - mx) / total;"),
    ("renorm_flag_ignored",
     "w[j] = renorm ? (exp((double)s[j].logit - mx) / total) / picked : exp((double)s[j].logit - mx) / total;",
     "w[j] = (exp((double)s[j].logit - mx) / total) / picked;"),
    ("shared_gate_not_applied", "const double c = shared_w ? shared_w[n] : 1.0;", "const double c = 1.0;"),
    ("silu_of_up", "hbuf[i] = gsum / (1.0 + exp(-gsum)) * usum;", "hbuf[i] = usum / (1.0 + exp(-usum)) * gsum;"),
    ("tokens_reversed_in_expert", "for (int32_t t = 0; t < T; ++t) {\n        for (int32_t j = 0; j < k; ++j) {\n            int32_t e = idx",
     "for (int32_t t = T - 1; t >= 0; --t) {\n        for (int32_t j = 0; j < k; ++j) {\n            int32_t e = idx"),
    ("shared_expert_dropped", "        if (has_shared) {\n            const double c",
     "        if (0) {\n            const double c"),
    ("down_reads_gate_scales", "osum += hbuf[i] * dequant_one(W->qd, W->sd, W->bd, row, I, G, i);",
     "osum += hbuf[i] * dequant_one(W->qd, W->sd, W->sd, row, I, G, i);"),
    ("rms_mean_over_h_minus_1", "const double inv = 1.0 / sqrt(ss / (double)H + eps);",
     "const double inv = 1.0 / sqrt(ss / (double)(H - 1) + eps);"),
    ("rms_eps_dropped", "const double inv = 1.0 / sqrt(ss / (double)H + eps);",
     "const double inv = 1.0 / sqrt(ss / (double)H);"),
    ("norm_weight_ignored", "x[o + k] = bf16_from_double((double)float_from_bf16(h[o + k]) * inv * (double)w[k]);",
     "x[o + k] = bf16_from_double((double)float_from_bf16(h[o + k]) * inv);"),
    ("residual_out_drops_h", "out[i] = bf16_from_double((double)float_from_bf16(h[i]) + y[i]);",
     "out[i] = bf16_from_double(y[i]);"),
    ("double_rounding_to_bf16", "return bf16_from_float((float)ldexp(r, e - 8));",
     "return bf16_from_float((float)v);"),
    ("attention_heads_interleaved", "const int32_t g = h / group;", "const int32_t g = h % Hkv;"),
    ("attention_scale_dropped", "s[t] = scale * acc;", "s[t] = acc;"),
    ("attention_not_normalised", "o[(int64_t)h * D + d] = acc / sum;", "o[(int64_t)h * D + d] = acc;"),
    ("attention_misses_last_position", "        for (int32_t t = 0; t < L; ++t) {\n            double acc = 0.0;",
     "        for (int32_t t = 0; t < L - 1; ++t) {\n            double acc = 0.0;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: anchor not found once"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(mutant_c), "-o", str(so), "-lm"])
    env = dict(os.environ, MOE_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"the pins did not catch the planted mistake {name}:\n{r.stdout[-2000:]}"


def test_unmodified_copy_passes(tmp_path):
    """Control: the same build-and-load route with the source unchanged passes
    every pin (so a failing mutant fails because of its mistake)."""
    so = tmp_path / "libcopy.so"
    subprocess.check_call(["gcc", *oracle.CFLAGS, SRC, "-o", str(so), "-lm"])
    env = dict(os.environ, MOE_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]

"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each case below plants one mistake (a dropped term, a wrong sign, a wrong
operand or index, a swapped order) in a copy of ``oracle/gdn_oracle.c``,
builds it with gcc into a temporary directory, and runs the pin suite against
that build in a child process.  The pin suite must fail for every mutant.
The real oracle source is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

MUTANTS = {
    "delta_sign": ("delta = beta * (v[i] - pred);", "delta = beta * (v[i] + pred);"),
    "no_decay": ("row[j] *= alpha;", "row[j] *= 1.0;"),
    "predict_with_query": ("pred += row[j] * k[j];", "pred += row[j] * q[j];"),
    "read_with_key": ("out += row[j] * q[j];", "out += row[j] * k[j];"),
    "read_before_correct": (
        "for (int j = 0; j < Dk; ++j) row[j] += delta * k[j];    /* correct */\n"
        "    double out = 0.0;\n"
        "    for (int j = 0; j < Dk; ++j) out += row[j] * q[j];      /* read    */",
        "double out = 0.0;\n"
        "    for (int j = 0; j < Dk; ++j) out += row[j] * q[j];      /* read    */\n"
        "    for (int j = 0; j < Dk; ++j) row[j] += delta * k[j];    /* correct */"),
    "predict_before_decay": (
        "for (int j = 0; j < Dk; ++j) row[j] *= alpha;          /* decay   */\n"
        "    double pred = 0.0;\n"
        "    for (int j = 0; j < Dk; ++j) pred += row[j] * k[j];     /* predict */",
        "double pred = 0.0;\n"
        "    for (int j = 0; j < Dk; ++j) pred += row[j] * k[j];     /* predict */\n"
        "    for (int j = 0; j < Dk; ++j) row[j] *= alpha;          /* decay   */"),
    "l2_no_eps": ("double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / sqrt(ss);"),
    "norm_sum_not_mean": ("sqrt(ss / n + eps)", "sqrt(ss + eps)"),
    "norm_no_silu_gate": ("* oracle_silu(z[i]);", "* z[i];"),
    "norm_one_plus_w": ("y[i] = w[i] * (x[i] * inv)", "y[i] = (1.0 + w[i]) * (x[i] * inv)"),
    "conv_taps_reversed": ("acc += taps[j] * window[j];", "acc += taps[3 - j] * window[j];"),
    "conv_no_silu": ("return oracle_silu(acc);", "return acc;"),
    "head_map_modulo": ("kh = h / r;", "kh = h % s->Hk;"),
    "k_reads_q_channels": ("return (size_t)s->Hk * s->Dk + (size_t)kh * s->Dk + i;",
                           "return (size_t)kh * s->Dk + i;"),
    "no_query_scale": ("oracle_l2norm(Dk, qraw, s->eps_l2, s->q_scale, qh);",
                       "oracle_l2norm(Dk, qraw, s->eps_l2, 1.0, qh);"),
    "window_newest_first": ("conv0[((size_t)b * 3 + e) * C + c]",
                            "conv0[((size_t)b * 3 + (2 - e)) * C + c]"),
    "carried_window_off_by_one": ("xext(s, qkv_pre, conv0, b, T + e, c);",
                                  "xext(s, qkv_pre, conv0, b, T + e - 1, c);"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "softplus_drops_linear_term": ("x > 0.0 ? x + log1p(exp(-x))", "x > 0.0 ? log1p(exp(-x))"),
    "decay_A_log_not_exponentiated": ("*g = -exp(A_log) *", "*g = -A_log *"),
    "decay_no_dt_bias": ("oracle_softplus(a + dt_bias)", "oracle_softplus(a)"),
    "write_gate_from_a": ("*beta = oracle_sigmoid(b);", "*beta = oracle_sigmoid(a);"),
    "gate_parameters_of_head_zero": ("(double)raw->A_log[h],\n                     (double)raw->dt_bias[h]",
                                     "(double)raw->A_log[0],\n                     (double)raw->dt_bias[0]"),
    "snapshots_reversed": ("S_snap + ((size_t)u * T + t) * Dv * Dk",
                           "S_snap + ((size_t)u * T + (T - 1 - t)) * Dv * Dk"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site for %r not found exactly once" % name
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", "-o", str(lib), str(mut), "-lm"], check=True)
    env = dict(os.environ, GDN_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, "pins did not catch mutant %r:\n%s" % (name, r.stdout[-2000:])

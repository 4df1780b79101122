"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a temporary copy of oracle/oracle.c (a dropped term, a wrong sign,
a transposed or shifted index, a wrong slot), builds it, and runs the pin
suite (tests/test_oracle_pins.py) against that build in a subprocess: the suite
must fail.  CPU only; nothing here touches a GPU."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "oracle", "oracle.c")).read()

MUTATIONS = {
    "beta_dropped": ("S[kk * V + vv] += kh[kk] * (bt * (vt[vv] - u[vv]));",
                     "S[kk * V + vv] += kh[kk] * ((vt[vv] - u[vv]));"),
    "delta_sign": ("(bt * (vt[vv] - u[vv]))", "(bt * (u[vv] - vt[vv]))"),
    "readout_before_decay": ("/* S <- exp(g) * S, row kk scaled by exp(g_kk) */",
                             "for (int64_t vv = 0; vv < V; ++vv) { double a = 0; for (int64_t kk = 0; kk < K; ++kk)"
                             " a += S[kk * V + vv] * kh[kk]; u[vv] = a; } if (0)"),
    "state_transposed": ("pool_get(pool, pool_bf16, st, r, hv, vv, kk)",
                         "pool_get(pool, pool_bf16, st, r, hv, kk % V, vv % K)"),
    "output_uses_k": ("acc += S[kk * V + vv] * qh[kk];", "acc += S[kk * V + vv] * kh[kk];"),
    "gqa_map": ("const int64_t h = hv / group;", "const int64_t h = hv % H;"),
    "softplus_bias_sign": ("x = -exp(A_log[hv]) * softplus(x + bias);", "x = -exp(A_log[hv]) * softplus(x - bias);"),
    "a_log_not_exponentiated": ("x = -exp(A_log[hv]) * softplus(x + bias);", "x = -A_log[hv] * softplus(x + bias);"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "l2_eps_outside_sqrt": ("const double nq = sqrt(sq + 1e-6), nk = sqrt(sk + 1e-6);",
                            "const double nq = sqrt(sq) + 1e-6, nk = sqrt(sk) + 1e-6;"),
    "la_decay_dropped": ("S[kk * V + vv] = lam * S[kk * V + vv] + kt[kk] * vt[vv];",
                         "S[kk * V + vv] = S[kk * V + vv] + kt[kk] * vt[vv];"),
    "la_row_index": ("const int64_t row = r * H + h;", "const int64_t row = r + h * P;"),
    "scale_dropped": ("out[((b * T + t) * HV + hv) * V + vv] = scale * acc;",
                      "out[((b * T + t) * HV + hv) * V + vv] = acc;"),
    "cache_shifted": ("if (tok) {\n                    double* it = tok + (((b * T + t) * HV + hv) * V) * K;",
                      "if (tok && t > 0) {\n                    double* it = tok + (((b * T + t - 1) * HV + hv) * V) * K;"),
    "kda_channel_reversed": ("dt_bias[hv * K + kk]", "dt_bias[hv * K + (K - 1 - kk)]"),
    "negative_write_not_skipped": ("        const int64_t w = write_idx ? write_idx[b] : read_idx[b];\n"
                                   "        if (w < 0) continue;\n        if (w >= P) { ++bad; continue; }\n"
                                   "        for (int64_t hv",
                                   "        int64_t w = write_idx ? write_idx[b] : read_idx[b];\n"
                                   "        if (w < 0) w = 0;\n        if (w >= P) { ++bad; continue; }\n"
                                   "        for (int64_t hv"),
    "empty_span_not_written": ("        if (w < 0) continue;\n        if (w >= P) { ++bad; continue; }\n"
                               "        for (int64_t hv",
                               "        if (w < 0 || T == 0) continue;\n        if (w >= P) { ++bad; continue; }\n"
                               "        for (int64_t hv"),
    "bf16_truncates": ("const double r = nearbyint(ax / q) * q;", "const double r = floor(ax / q) * q;"),
    "seed_off_by_one": ("r = state_idx[b * T + a - 1];", "r = state_idx[b * T + (a < T ? a : a - 1)];"),
    "token_state_shifted": ("const double* f = tok + (((b * T + t) * HV + hv) * V) * K;",
                            "const double* f = tok + (((b * T + (t > 0 ? t - 1 : t)) * HV + hv) * V) * K;"),
}


def _run_pins(source: str, tmp_path):
    src = tmp_path / "oracle.c"
    src.write_text(source)
    lib = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(lib), str(src), "-lm"])
    env = dict(os.environ, LAR_ORACLE_LIB=str(lib))
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                           os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_control_unmodified_source_passes(tmp_path):
    r = _run_pins(SRC, tmp_path)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path):
    old, new = MUTATIONS[name]
    assert SRC.count(old) >= 1, f"mutation site for {name} not found"
    r = _run_pins(SRC.replace(old, new, 1), tmp_path)
    assert r.returncode != 0, f"mutation {name} survived the pins:\n{r.stdout[-1500:]}"

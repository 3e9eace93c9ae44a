"""The oracle's pins catch plausible mistakes (CPU only).

Each case copies the oracle and its pin tests into a temporary directory,
plants one mistake in the copied C source, and runs the pins there: they must
fail.  The real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("philox key xor dropped", "uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;",
     "uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1;"),
    ("nine Philox rounds", "for (int round = 0; round < 10; ++round)",
     "for (int round = 0; round < 9; ++round)"),
    ("uniform off by one step", "return ((double)(w >> 9) * 2.0 + 1.0) * 0x1p-24;",
     "return ((double)(w >> 9) * 2.0 + 2.0) * 0x1p-24;"),
    ("anchor ignored", "  int32_t prev = J->x0[i];\n  for (int k = 1;", "  int32_t prev = 0;\n  for (int k = 1;"),
    ("previous token not advanced", "oracle_markov_bias(J->W1, J->W2, J->V, J->r, prev, s);\n    prev = draft_sample(",
     "oracle_markov_bias(J->W1, J->W2, J->V, J->r, prev, s);\n    (void)draft_sample("),
    ("temperature dropped", "s[v] = (Uk[v] + s[v]) / J->T;", "s[v] = (Uk[v] + s[v]);"),
    ("bias sign", "out[v] += a * w2row[v];", "out[v] -= a * w2row[v];"),
    ("accept comparison reversed", "if (!((float)lhs < (float)rhs)) break;",
     "if (!((float)lhs > (float)rhs)) break;"),
    ("residual sign", "const double res = pt - pd;", "const double res = pd - pt;"),
    ("emitted token is the rejected draft", "t[n] = tok;",
     "t[n] = J->x[(size_t)i * g + (n < g ? n : g - 1)];"),
    ("max instead of min in c*", "cs += pd < pt ? pd : pt;", "cs += pd > pt ? pd : pt;"),
    ("scheduler never stops", "if (!exact_greater(tau_i, sps[B + 1], tau, sps[B])) break;",
     "if (0) break;"),
    ("scheduler comparison reversed", "if (!exact_greater(tau_i, sps[B + 1], tau, sps[B])) break;",
     "if (!exact_greater(tau, sps[B], tau_i, sps[B + 1])) break;"),
    ("step rate of the wrong batch size", "if (!exact_greater(tau_i, sps[B + 1], tau, sps[B])) break;",
     "if (!exact_greater(tau_i, sps[B], tau, sps[B])) break;"),
    ("survival not a product", "a = (j == 0) ? cj : a * cj;", "a = cj;"),
    ("bonus row one too early", "const int row = L + 1;", "const int row = L > 0 ? L : 1;"),
    ("capacity keeps Algorithm 1's early stop",
     "if (exact_greater(tau, sps[R + i + 1], best_tau, sps[R + best])) { /* strictly: first maximum */",
     "if (!exact_greater(tau, sps[R + i + 1], best_tau, sps[R + best])) break;\n    { /* strictly: first maximum */"),
    ("capacity reads the step rate one batch early",
     "if (exact_greater(tau, sps[R + i + 1], best_tau, sps[R + best])) { /* strictly: first maximum */",
     "if (exact_greater(tau, sps[R + i], best_tau, sps[R + best])) { /* strictly: first maximum */"),
    ("top-k takes one candidate too many", "for (int i = 0; i < n && i < K; ++i) ell[cs[i].r] += 1;",
     "for (int i = 0; i < n && i <= K; ++i) ell[cs[i].r] += 1;"),
    ("temperature multiplies the logit", "const double z = (log(c) - log1p(-c)) / T;",
     "const double z = (log(c) - log1p(-c)) * T;"),
    ("ECE without the absolute value",
     "      double e = 0.0;\n      for (int b = 0; b < M; ++b) e += fabs(bins[b]);\n      e /= (double)N;",
     "      double e = 0.0;\n      for (int b = 0; b < M; ++b) e += bins[b];\n      e /= (double)N;"),
    ("ECE bins one short", "        int b = (int)floor(a * M);", "        int b = (int)floor(a * (M - 1));"),
    ("earlier positions' calibration not kept",
     "      ahat[s] *= oracle_temper((double)c[(size_t)s * gamma + k], grid[best]);",
     "      ahat[s] *= 1.0;"),
    ("threshold test strict", "if (!(a >= theta)) break;", "if (!(a > theta)) break;"),
    ("RNN head without the tanh", "      hn[j] = tanh(z);", "      hn[j] = z;"),
    ("RNN state not carried", "      h[j] = hn[j];", "      h[j] = 0.0;"),
    ("RNN recurrent matrix transposed", "for (int a = 0; a < r; ++a) z += h[a] * Wh[(size_t)a * r + j];",
     "for (int a = 0; a < r; ++a) z += h[a] * Wh[(size_t)j * r + a];"),
    ("RNN operand not rounded to bf16", "      A[j] = oracle_round_bf16(hn[j]);", "      A[j] = hn[j];"),
    ("draft stream keyed by the wrong position",
     "two_level_argmax(s, V, J->seed, req, (uint32_t)k, ORACLE_PURPOSE_DRAFT_GROUP,",
     "two_level_argmax(s, V, J->seed, req, (uint32_t)(k + 1), ORACLE_PURPOSE_DRAFT_GROUP,"),
    ("group mass is the group's largest weight",
     "gkey[j] = (m + log(t)) + oracle_gumbel(", "gkey[j] = m + oracle_gumbel("),
    ("second stage searches the first group",
     "const int a = j * ORACLE_GROUP, n =", "const int a = 0 * ORACLE_GROUP, n ="),
    ("group draws keyed like the id draws",
     "ORACLE_PURPOSE_DRAFT_GROUP,\n                                  ORACLE_PURPOSE_DRAFT, key, &margin);",
     "ORACLE_PURPOSE_DRAFT,\n                                  ORACLE_PURPOSE_DRAFT, key, &margin);"),
    ("RNN anchor ignored", "  int32_t prev = J->x0[i];\n  double* h", "  int32_t prev = 0;\n  double* h"),
    ("RNN previous token not advanced", "    }\n    prev = draft_sample(J, i, k, s, key);",
     "    }\n    (void)draft_sample(J, i, k, s, key);"),
]


def _prepare(tmp):
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(tmp, "oracle"),
                    ignore=shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__"))
    os.makedirs(os.path.join(tmp, "tests"))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(tmp, "tests", "golden"))
    for f in os.listdir(os.path.join(ROOT, "tests")):
        if f.startswith("test_oracle_") and f.endswith(".py") and f != os.path.basename(__file__):
            shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(tmp, "tests", f))
    shutil.copy(os.path.join(ROOT, "tests", "conftest.py"), os.path.join(tmp, "tests", "conftest.py"))


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    tmp = str(tmp_path)
    _prepare(tmp)
    src = os.path.join(tmp, "oracle", "dspark_oracle.c")
    text = open(src).read()
    assert text.count(old) == 1, f"mutation site not found: {old!r}"
    open(src, "w").write(text.replace(old, new))
    env = dict(os.environ, PYTHONPATH=tmp, PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests", "-x", "-q", "-p", "no:cacheprovider",
                        "-k", "not mutation"], cwd=tmp, env=env, capture_output=True, text=True,
                       timeout=900)
    assert "libdspark_oracle" not in r.stderr or r.returncode != 0
    assert r.returncode != 0, f"pins passed with the mistake '{name}' planted:\n{r.stdout[-500:]}"
    assert "failed" in r.stdout, r.stdout[-800:] + r.stderr[-800:]

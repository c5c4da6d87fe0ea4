"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, a wrong index, a transposed operand, an exclusive prefix,
the wrong routing rows), builds the copy, and runs the pins of
test_oracle_pins.py against it in a child process.  The drift guard (values
recorded from the oracle itself) is left out, so a mutant only fails through
a pin that is independent of the oracle.  A mutant that every pin lets
through fails this test.
"""
import os
import subprocess
import sys

import pytest

import oracle

# several pins compare with scikit-learn's GMM posterior; without it some mutants would
# only be caught by the drift guard, which is left out here
pytest.importorskip("sklearn")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

CAUSAL_STEP = """            posterior(d, K, mu_h, var_h, lp_h, kx + ((long)s * N + i) * d, g, ll);
            write_row(K, dv, g, v + ((long)s * N + i) * dv, Vt, Z);
            posterior(d, K, mu_h, var_h, lp_h, qx + ((long)s * N + i) * d, g, ll);
            read_row(K, dv, g, Vt, Z, eps, out + ((long)s * N + i) * dv);"""
BIDIR_READ = """            posterior(d, K, mu_h, var_h, lp_h, qx + ((long)s * N + i) * d, g, ll);
            read_row(K, dv, g, Vt, Z, eps, out + ((long)s * N + i) * dv);
        }
        free(Vt);"""

# (what the mistake is, text in the oracle, replacement, replace every occurrence)
MUTANTS = [
    ("S0 softplus without its branch for negative r",
     "return fmax(r, 0.0) + log1p(exp(-fabs(r)));", "return fmax(r, 0.0) + log1p(exp(-r));", False),
    ("S0 raw variances used without softplus",
     "var[i] = softplus(var_raw[i]);", "var[i] = fabs(var_raw[i]) + 1e-3;", False),
    ("S0 log-sum-exp of the logits without the max shift",
     "for (int k = 0; k < K; ++k) s += exp(l[k] - m);", "for (int k = 0; k < K; ++k) s += exp(l[k]);", False),
    ("S1 log-variance term dropped",
     "q += t * t / vk[j] + log(vk[j]) + kLog2Pi;", "q += t * t / vk[j] + kLog2Pi;", False),
    ("S1 multiplied by the variance instead of divided",
     "q += t * t / vk[j] + log(vk[j]) + kLog2Pi;", "q += t * t * vk[j] + log(vk[j]) + kLog2Pi;", False),
    ("S1 prior with the wrong sign",
     "ll[k] = log_pi[k] - 0.5 * q;", "ll[k] = -log_pi[k] - 0.5 * q;", False),
    ("S1 factor one half dropped",
     "ll[k] = log_pi[k] - 0.5 * q;", "ll[k] = log_pi[k] - q;", False),
    ("S1 posterior not normalised",
     "for (int k = 0; k < K; ++k) gamma[k] /= den;", "for (int k = 0; k < K; ++k) gamma[k] /= 1.0;", False),
    ("S1 every slice routed with head 0",
     "int h = head[s];", "int h = 0 * head[s];", True),
    ("S2 normaliser Z not accumulated",
     "        Z[k] += gk[k];", "        Z[k] += 0.0 * gk[k];", False),
    ("S2 value column index shifted",
     "for (int c = 0; c < dv; ++c) Vt[(long)k * dv + c] += gk[k] * v[c];",
     "for (int c = 0; c < dv; ++c) Vt[(long)k * dv + c] += gk[k] * v[(c + 1) % dv];", False),
    ("S3 denominator reads one slot of Z",
     "for (int k = 0; k < K; ++k) den += gq[k] * Z[k];", "for (int k = 0; k < K; ++k) den += gq[k] * Z[0];", False),
    ("S3 eps dropped from the denominator",
     "    den += eps;\n", "    den += 0.0 * eps;\n", False),
    ("S3 latent memory read transposed",
     "for (int k = 0; k < K; ++k) num += gq[k] * Vt[(long)k * dv + c];",
     "for (int k = 0; k < K; ++k) num += gq[k] * Vt[(long)c * K + k];", False),
    ("S3 bidirectional read routes the key rows",
     BIDIR_READ, BIDIR_READ.replace("qx + ((long)s", "kx + ((long)s"), False),
    ("S4 exclusive prefix (read before write)",
     CAUSAL_STEP, "\n".join(CAUSAL_STEP.split("\n")[2:] + CAUSAL_STEP.split("\n")[:2]), False),
    ("S4 causal write routes the query rows",
     CAUSAL_STEP, CAUSAL_STEP.replace("kx + ((long)s", "qx + ((long)s"), False),
    ("S4/S5 incoming state ignored",
     "        if (state_in) memcpy(st, state_in + s * sz, sizeof(double) * (size_t)sz);\n", "", False),
    ("X cross-attention writes only the first key row",
     "for (int j = 0; j < Nk; ++j) {", "for (int j = 0; j < (Nk > 0 ? 1 : 0); ++j) {", False),
    ("G denominator gradient with the wrong sign",
     "    ui[dv] = -go / den;", "    ui[dv] = go / den;", False),
    ("G softmax backward without the row term",
     "const double delta = g[(long)i * K + k] * (dg[(long)i * K + k] - dot);",
     "const double delta = g[(long)i * K + k] * dg[(long)i * K + k];", False),
    ("G causal key side summed over the prefix instead of the suffix",
     "        for (int j = N - 1; j >= 0; --j) {", "        for (int j = 0; j < N; ++j) {", False),
    ("G softplus derivative dropped",
     "dvar_raw[e] *= 1.0 / (1.0 + exp(-var_raw[e]));", "dvar_raw[e] *= 1.0;", False),
    ("G logit gradient from the query rows only",
     "                    plp[(long)s * K + k] += delta;", "                    if (!pass) plp[(long)s * K + k] += delta;",
     False),
    ("G variance gradient without the log-determinant term",
     "delta * (0.5 * t * t / (sk * sk) - 0.5 / sk);", "delta * (0.5 * t * t / (sk * sk));", False),
    ("G value gradient from the query responsibilities",
     "for (int k = 0; k < K; ++k) t += gk[(long)j * K + k] * M[k * w + c];",
     "for (int k = 0; k < K; ++k) t += gq[(long)j * K + k] * M[k * w + c];", False),
    ("D ties assigned to the highest component",
     "if (g[k] > g[best]) best = k;", "if (g[k] >= g[best]) best = k;", False),
    ("D soft usage sums the squared posterior",
     "usage[(long)h * K + k] += g[k];", "usage[(long)h * K + k] += g[k] * g[k];", False),
    ("D every head's usage accumulated on head 0",
     "usage[(long)h * K + k] += g[k];", "usage[k] += g[k];", False),
    ("D entropy not divided by log K",
     "return h / log((double)K);", "return h;", False),
    ("D hard-assignment entropy taken from the soft usage",
     "entropy[2 * h + 1] = normalised_entropy(K, w);",
     "entropy[2 * h + 1] = normalised_entropy(K, usage + (long)h * K);", False),
]


@pytest.mark.parametrize("what,old,new,every", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(tmp_path, what, old, new, every):
    src = open(oracle._SRC).read()
    n = src.count(old)
    assert n >= 1 and (every or n == 1), f"{what}: the text to mutate occurs {n} times"
    mutated = src.replace(old, new)
    assert mutated != src
    c = tmp_path / "mutant.c"
    c.write_text(mutated)
    lib = tmp_path / "libmutant.so"
    oracle.compile_to(str(c), str(lib))
    env = dict(os.environ, GMA_ORACLE_LIB=str(lib), OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider",
                        "-k", "not recorded_values"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    # exit status 1: some pin failed; 0 would mean the mistake went through every pin
    assert r.returncode == 1, f"{what}: pins exit {r.returncode}\n{r.stdout[-3000:]}"
    assert "failed" in r.stdout


def test_a_change_that_is_not_a_mistake_goes_through(tmp_path):
    """Control: dropping the log(2 pi) constant, which cancels in the posterior, changes
    no result beyond rounding, and every pin passes on that build."""
    src = open(oracle._SRC).read()
    old = "q += t * t / vk[j] + log(vk[j]) + kLog2Pi;"
    assert src.count(old) == 1
    c = tmp_path / "same.c"
    c.write_text(src.replace(old, "q += t * t / vk[j] + log(vk[j]);"))
    lib = tmp_path / "libsame.so"
    oracle.compile_to(str(c), str(lib))
    env = dict(os.environ, GMA_ORACLE_LIB=str(lib), OMP_NUM_THREADS="4")
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-q", "-p", "no:cacheprovider",
                        "-k", "not recorded_values"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-3000:]

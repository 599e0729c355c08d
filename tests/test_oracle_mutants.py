"""Plants plausible mistakes in the oracle (on the CPU) and checks that the pin
suite catches each one.

Each mutant is a one-line textual edit of a copy of ``oracle/gdn_oracle.c``.
The copy is compiled with gcc into a temporary directory. The pin suite then
runs against it in a child pytest, and must fail there. This test shows that
the pins constrain every step of the oracle, not only its composition.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

# (name, original text, replacement, replace every occurrence)
MUTANTS = [
    ("decay_sign", "double a = exp(g);", "double a = exp(-g);", False),
    ("no_decay", "for (size_t e = 0; e < (size_t)dk * dv; ++e) S[e] *= a;", "(void)a;", False),
    ("delta_sign", "double delta = (v[j] - pred) * b;", "double delta = (v[j] + pred) * b;", False),
    ("no_beta", "double delta = (v[j] - pred) * b;", "double delta = (v[j] - pred);", False),
    ("no_write", "S[(size_t)i * dv + j] += k[i] * delta;", "(void)delta;", False),
    ("scale_twice", "y[j] = scale * acc;", "y[j] = scale * scale * acc;", False),
    ("blocked_gqa", "int kh = vh % d->Hk;", "int kh = vh / (d->Hv / d->Hk);", True),
    ("conv_taps_reversed", "u += w[(size_t)c * Kc + m] * state[(size_t)m * C + c];",
     "u += w[(size_t)c * Kc + m] * state[(size_t)(Kc - 2 - m) * C + c];", False),
    ("conv_current_tap0", "u += w[(size_t)c * Kc + (Kc - 1)] * x[c];", "u += w[(size_t)c * Kc] * x[c];",
     False),
    ("conv_push_front", "state[(size_t)(Kc - 2) * C + c] = x[c];", "state[c] = x[c];", False),
    ("l2_is_rms", "double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / sqrt(ss / n + eps);", False),
    ("gate_sigmoid", "out[j] = y[j] * r * w[j] * silu(z[j]);",
     "out[j] = y[j] * r * w[j] * (1.0 / (1.0 + exp(-z[j])));", False),
    ("norm_one_plus_w", "out[j] = y[j] * r * w[j] * silu(z[j]);",
     "out[j] = y[j] * r * (1.0 + w[j]) * silu(z[j]);", False),
    ("softplus_no_one", "x > 20.0 ? x : log1p(exp(x))", "x > 20.0 ? x : log(exp(x))", False),
    ("beta_sign", "*b_out = 1.0 / (1.0 + exp(-beta));", "*b_out = 1.0 / (1.0 + exp(beta));", False),
    ("q_k_swapped", "const double *q = xhat + (size_t)kh * d->dk;",
     "const double *q = xhat + (size_t)d->Hk * d->dk + (size_t)kh * d->dk;", True),
    ("chunk_L_exponent", "val = exp(G[r] - G[s]) * dot;", "val = exp(G[s] - G[r]) * dot;", False),
    ("chunk_no_diagonal", "for (int s = 0; s <= r; ++s) {", "for (int s = 0; s < r; ++s) {", False),
    ("chunk_update_decay", "upd += K[(size_t)s * dk + i] * exp(G[n - 1] - G[s]) * Vn[(size_t)s * dv + j];",
     "upd += K[(size_t)s * dk + i] * Vn[(size_t)s * dv + j];", False),
]


def test_mutant_table_applies():
    src = open(SRC).read()
    for name, old, new, _ in MUTANTS:
        assert old in src, f"mutant {name}: pattern not found in the oracle source"


@pytest.mark.parametrize("name,old,new,every", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, name, old, new, every):
    src = open(SRC).read()
    mutated = src.replace(old, new) if every else src.replace(old, new, 1)
    assert mutated != src
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "libmutant.so"
    c_path.write_text(mutated)
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-o", str(so_path),
                           str(c_path), "-lm"])
    env = dict(os.environ, GDN_ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pin suite:\n{r.stdout[-2000:]}"

"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is a copy of oracle/gdn_oracle.c with one passage replaced by a
plausible mistake, compiled like the oracle into a temporary directory.  The
oracle source itself carries none of them.  Every planted edit must match the
source exactly once, so the list cannot drift away from the oracle unnoticed.
CPU only.
"""
import os

import pytest

import oracle as O
import oracle_pins as P

I16, I20 = " " * 16, " " * 20

_O_LOOP = (f"{I16}for (int r = 0; r < d; ++r) {{\n"
           f"{I20}double acc = 0.0;\n"
           f"{I20}for (int c = 0; c < d; ++c) acc += S[(size_t)r * d + c] * qn[c];\n"
           f"{I20}orow[r] = q_scale * acc;\n"
           f"{I16}}}\n")
_UPDATE = (f"{I16}for (int r = 0; r < d; ++r)\n"
           f"{I20}for (int c = 0; c < d; ++c) S[(size_t)r * d + c] += u[r] * kn[c];\n")

# (what the mistake is, correct passage, planted passage)
MUTANTS = [
    ("conv taps reversed",
     "acc += (double)col[K - 1 - j][c] * (double)conv_w[(size_t)c * K + j];",
     "acc += (double)col[K - 1 - j][c] * (double)conv_w[(size_t)c * K + (K - 1 - j)];"),
    ("history order flipped",
     "col[b] = hist + (size_t)(K - 2 - above) * C;",
     "col[b] = hist + (size_t)above * C;"),
    ("decay dropped",
     "S[e] = decay * Sp[e];",
     "S[e] = Sp[e];"),
    ("sign of the delta flipped",
     "u[r] = beta * ((double)v[r] - sk);",
     "u[r] = beta * (sk - (double)v[r]);"),
    ("state read transposed",
     "S0[(size_t)r * d + c] = S0f[(size_t)r * d + c];",
     "S0[(size_t)r * d + c] = S0f[(size_t)c * d + r];"),
    ("grouped heads mapped h mod H_k",
     "const int kh = h / G;                  /* [P3] q/k heads broadcast */",
     "const int kh = h % Hk;"),
    ("output read before the rank-one update",
     _UPDATE + _O_LOOP,
     _O_LOOP + _UPDATE),
    ("k not normalised",
     "l2_normalise(k, kn, d);",
     "for (int c = 0; c < d; ++c) kn[c] = k[c];"),
    ("dt_bias dropped",
     "exp(softplus(a + (double)dt_bias[h]) * (double)A[h]);",
     "exp(softplus(a) * (double)A[h]);"),
    ("commit path applied leaf first",
     "const int j = path[m - 1 - step];",
     "const int j = path[step];"),
    ("commit window taken from the parent",
     "const int wnode = a;",
     "const int wnode = parents[n0 + a] >= 0 ? parents[n0 + a] : a;"),
    ("b and a swapped",
     "const double b = ba[(size_t)t * ba_stride + h];\n"
     f"{I16}const double a = ba[(size_t)t * ba_stride + Hv + h];",
     "const double b = ba[(size_t)t * ba_stride + Hv + h];\n"
     f"{I16}const double a = ba[(size_t)t * ba_stride + h];"),
    ("SiLU dropped",
     "xc[(size_t)(n0 + i) * C + c] = silu(acc);",
     "xc[(size_t)(n0 + i) * C + c] = acc;"),
    ("q not normalised",
     "l2_normalise(q, qn, d);",
     "for (int c = 0; c < d; ++c) qn[c] = q[c];"),
]


@pytest.fixture(scope="module")
def oracle_source():
    with open(O.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("what,good,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(what, good, bad, oracle_source, tmp_path):
    assert oracle_source.count(good) == 1, f"planted edit '{what}' no longer matches the oracle"
    src = tmp_path / "gdn_oracle_mutant.c"
    src.write_text(oracle_source.replace(good, bad))
    lib = O.compile_source(str(src), str(tmp_path / "liboracle_mutant.so"))
    orc = O.Oracle(lib_path=lib)
    caught = []
    for check in P.ALL_CHECKS:
        try:
            check(orc)
        except AssertionError:
            caught.append(check.__name__)
    assert caught, f"mutant '{what}' passed every pin"
    assert os.path.exists(lib)

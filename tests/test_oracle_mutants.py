"""The oracle pins must fail on plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, and checks that the decimal brute force
or a closed form rejects it.  Nothing here touches the GPU or the product.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from test_oracle_pins import _brute_prefill

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle",
                   "parallax_oracle.c")

MUTANTS = {
    "sign_flip": ("C[a * d + c];\n            out[c] = mu_v[c] - corr;",
                  "C[a * d + c];\n            out[c] = mu_v[c] + corr;"),
    "transposed_cov": ("corr += rho[a] * C[a * d + c];", "corr += rho[a] * C[c * d + a];"),
    # (dropping the centering of only one side would NOT be a mistake: the
    # weighted mean of (v - mu_v) is zero, so either centering suffices)
    "unweighted_cov": ("double ka = p[j] * (K[j * d + a] - mu_k[a]);",
                       "double ka = (K[j * d + a] - mu_k[a]);"),
    "contracted_sign": ("out[c] = mu_v[c] - corr;\n        }\n        return 0;\n    }\n    return -2;",
                        "out[c] = mu_v[c] + corr;\n        }\n        return 0;\n    }\n    return -2;"),
    "causal_off_by_one": ("const int64_t n = causal ? i + 1 : L;",
                          "const int64_t n = causal ? (i > 0 ? i : 1) : L;"),
    "scale_dropped": ("p[j] = scale * dot;\n        if (p[j] > mx) mx = p[j];\n    }\n    double z",
                      "p[j] = dot;\n        if (p[j] > mx) mx = p[j];\n    }\n    double z"),
    "uncentered_missing_mean_term": ("out[c] = mu - (W[c] / l - (A / l) * mu);",
                                     "out[c] = mu - W[c] / l;"),
}
FORM_OF = {"contracted_sign": 1, "uncentered_missing_mean_term": 2}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", str(lib), str(path), "-lm"],
                   check=True)
    return ctypes.CDLL(str(lib))


def _run(lib, q, rho, k, v, causal, scale, form):
    dp = ctypes.POINTER(ctypes.c_double)
    i64 = ctypes.c_int64
    lib.oracle_prefill.argtypes = [dp, dp, dp, dp, i64, i64, i64, i64, ctypes.c_int,
                                   ctypes.c_double, ctypes.c_int, dp]
    o = np.empty_like(q)
    p = lambda a: a.ctypes.data_as(dp)
    B, H, L, d = q.shape
    rc = lib.oracle_prefill(p(q), p(rho), p(k), p(v), B, H, L, d, int(causal), scale, form, p(o))
    assert rc == 0
    return o


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    rng = np.random.default_rng(99)
    q, rho, k, v = (np.ascontiguousarray(rng.standard_normal((1, 1, 5, 3))) for _ in range(4))
    ref = _brute_prefill(q, rho, k, v, True, 0.7)
    got = _run(lib, q, rho, k, v, True, 0.7, FORM_OF.get(name, 0))
    assert np.abs(got - ref).max() > 1e-6, f"mutant {name} slipped past the brute force"

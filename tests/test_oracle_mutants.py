"""Plant plausible mistakes in a COPY of the oracle and check that the pins
catch every one of them (CPU only; the real oracle is never modified)."""
import os
import tempfile

import pytest

import oracle
import pins

# (name, text in oracle.c, replacement)
MUTANTS = [
    ("query correction sign", "rotate(qi, qg, D, floor_div(i, g) - i, theta);\n                    int64_t jmax = i < Sk - 1 ? i : Sk - 1;\n                    double m",
     "rotate(qi, qg, D, i - floor_div(i, g), theta);\n                    int64_t jmax = i < Sk - 1 ? i : Sk - 1;\n                    double m"),
    ("key correction sign", "floor_div(j, g) - j", "j - floor_div(j, g)"),
    ("window boundary off by one", "(i - j < w) ?", "(i - j <= w) ?"),
    ("group rule uses s instead of s-1", "while ((s - 1) / g > L - 1)", "while (s / g > L - 1)"),
    ("rotation sign of second half", "y[d + h] = x1 * c + x0 * s;", "y[d + h] = x1 * c - x0 * s;"),
    ("frequency exponent", "pow(theta, -2.0 * (double)d / (double)D)", "pow(theta, -(double)d / (double)D)"),
    ("softmax scale", "const double tau = 1.0 / sqrt((double)D);\n\n    for (int64_t b = 0; b < B; b++) {\n        for (int64_t hk = 0; hk < Hkv; hk++) {\n            double *kg = grouped_keys(k, b, hk, Sk, Hkv, D, g, theta);\n            if (!kg) return -1;\n            int64_t nrow",
     "const double tau = 1.0 / (double)D;\n\n    for (int64_t b = 0; b < B; b++) {\n        for (int64_t hk = 0; hk < Hkv; hk++) {\n            double *kg = grouped_keys(k, b, hk, Sk, Hkv, D, g, theta);\n            if (!kg) return -1;\n            int64_t nrow"),
    ("lse without the max", "\n                    lse[(b * Hq + h) * Sq + r] = (jmax >= 0) ? m + log(Z) : -INFINITY;",
     "\n                    lse[(b * Hq + h) * Sq + r] = (jmax >= 0) ? log(Z) : -INFINITY;"),
    ("GQA head mapping", "int64_t r = t / grp, h = hk * grp + t % grp;\n                    int64_t i = qpos[r];\n                    const double *qi = q + ((b * Sq + r) * Hq + h) * D;\n                    rotate(qi, qg, D, floor_div(i, g) - i, theta);\n                    int64_t jmax = i < Sk - 1 ? i : Sk - 1;\n                    double m",
     "int64_t r = t / grp, h = hk + (t % grp) * Hkv;\n                    int64_t i = qpos[r];\n                    const double *qi = q + ((b * Sq + r) * Hq + h) * D;\n                    rotate(qi, qg, D, floor_div(i, g) - i, theta);\n                    int64_t jmax = i < Sk - 1 ? i : Sk - 1;\n                    double m"),
    ("diagonal dropped", "int64_t jmax = i < Sk - 1 ? i : Sk - 1;\n                    double m",
     "int64_t jmax = i - 1 < Sk - 1 ? i - 1 : Sk - 1;\n                    double m"),
    ("inclusion-exclusion sign", "(eL * oL[d] + eA * oA[d] - eW * oW[d]) / Z", "(eL * oL[d] + eA * oA[d] + eW * oW[d]) / Z"),
    ("three-pass window start", "int64_t jwin = i - w + 1;", "int64_t jwin = i - w;"),
    # the variants (per-query g, sliding window, query shift)
    ("per-query g ignored", "int64_t s_row = (flags & ORACLE_PER_QUERY_G) ? qpos[r] + 1 : s_len;",
     "int64_t s_row = s_len;"),
    ("per-query length off by one", "int64_t s_row = (flags & ORACLE_PER_QUERY_G) ? qpos[r] + 1 : s_len;",
     "int64_t s_row = (flags & ORACLE_PER_QUERY_G) ? qpos[r] : s_len;"),
    ("query shift sign", "rotate(qi, qg, D, floor_div(i, g) + shift - i, theta);",
     "rotate(qi, qg, D, floor_div(i, g) - shift - i, theta);"),
    ("shift rounds w/g up", "const int64_t shift = (flags & ORACLE_QUERY_SHIFT) ? w - w / g : 0;",
     "const int64_t shift = (flags & ORACLE_QUERY_SHIFT) ? w - (w + g - 1) / g : 0;"),
    ("shifted rule bound", "if ((s - 1) / g + (w - w / g) <= L - 1) return g;",
     "if ((s - 1) / g + (w - w / g) < L - 1) return g;"),
    ("sliding window keeps far keys", "} else if (flags & ORACLE_SLIDING) {", "} else if (0) {"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site not unique/found: {name}"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "mutant.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new))
        mutant = oracle.Oracle(oracle.compile_oracle(path, os.path.join(d, "libmutant.so")))
        failed = []
        for pin in pins.ALL_PINS:
            try:
                if pin is pins.pin_brute:
                    pin(mutant, sizes=range(1, 8))
                else:
                    pin(mutant)
            except (AssertionError, ValueError):
                failed.append(pin.__name__)
        assert failed, f"mutant '{name}' passed every pin"

"""The oracle's pins must reject plausible mistakes in the oracle itself.

Each mutant below plants one such mistake in a copy of the oracle's C source
(on the CPU, in a temporary directory), builds it, and runs the pin suite
against it in a subprocess; the suite must fail.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mla_oracle.c")

MUTANTS = {
    "drop_rope_term": ("s += bf16_to_f64(qr[d]) * bf16_to_f64(k[J->Dl + d]);", "s += 0.0;"),
    "value_from_wrong_offset": ("o[d] += w * bf16_to_f64(v[d]);",
                                "o[d] += w * bf16_to_f64(v[d + J->Dr]);"),
    "mask_bits_msb_first": ("return (int)((row[j >> 5] >> (j & 31)) & 1u);",
                            "return (int)((row[j >> 5] >> (31 - (j & 31))) & 1u);"),
    "mask_transposed": ("const uint32_t *row = J->mask + ((size_t)b * J->q + i) * words;\n"
                        "    return (int)((row[j >> 5] >> (j & 31)) & 1u);",
                        "const uint32_t *row = J->mask + ((size_t)b * J->q + j) * words;\n"
                        "    return (int)((row[i >> 5] >> (i & 31)) & 1u);"),
    "prefix_off_by_one": ("if (t < prefix)\n        return 1;", "if (t <= prefix)\n        return 1;"),
    "scale_dropped": ("return J->scale * s;", "return s;"),
    "lse_log2": ("J->lse[r] = m + log(l);", "J->lse[r] = m + log2(l);"),
    "combine_weight_sign": ("double w = exp(m[(size_t)s * nrows + r] - M);",
                            "double w = exp(M - m[(size_t)s * nrows + r]);"),
    "no_normalisation": ("o[d] /= l;", "o[d] /= 1.0;"),
    "draft_order_reversed": ("int j = t - prefix;", "int j = S - 1 - t;"),
    "row_index_swapped": ("int h = (int)(r % J->H);\n    int i = (int)((r / J->H) % J->q);",
                          "int i = (int)(r % J->q);\n    int h = (int)((r / J->q) % J->H);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not found: %s" % name
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "mla_oracle.c")
        with open(c, "w") as fh:
            fh.write(src.replace(old, new))
        so = os.path.join(d, "libmut.so")
        subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-I", os.path.join(ROOT, "oracle"), "-o", so, c, "-lm"])
        env = dict(os.environ, MLA_ORACLE_LIB=so)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode != 0, "pins accepted mutant %s:\n%s" % (name, r.stdout[-2000:])

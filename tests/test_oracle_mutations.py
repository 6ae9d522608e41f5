"""Planted mistakes: a copy of the oracle with one plausible bug must fail at
least one pin.  The mistake is planted in a temporary copy of the C source on
the CPU; the committed oracle is never modified."""
import os

import pytest

import oracle as ora
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(ora.oracle.__file__), "ct_oracle.c")

# (name, text in the oracle, replacement).  Every replacement keeps all
# memory accesses in bounds; only the arithmetic is wrong.
MUTATIONS = [
    ("padding_sign", "i2 * Ss[2] - Pp[2] + k2 * Dd[2]", "i2 * Ss[2] + Pp[2] + k2 * Dd[2]"),
    ("kernel_flipped", "xv * wk[(k0 * Kk[1] + k1) * Kk[2] + k2]",
     "xv * wk[((Kk[0] - 1 - k0) * Kk[1] + (Kk[1] - 1 - k1)) * Kk[2] + (Kk[2] - 1 - k2)]"),
    ("bias_dropped", "yo[t] += bias[oc];", "yo[t] += 0.0 * bias[oc];"),
    ("weight_operand_transposed", "const double *wk = w + (ic * Cog + ocl) * kvol;\n                double *yo",
     "const double *wk = w + (ocl * C_in + ic) * kvol;\n                double *yo"),
    ("group_mapping_dropped", "const int64_t oc = g * Cog + ocl;", "const int64_t oc = ocl;"),
    ("out_len_off_by_one", "+ dl * (k - 1) + op + 1;", "+ dl * (k - 1) + op;"),
    ("dilation_dropped", "i2 * Ss[2] - Pp[2] + k2 * Dd[2]", "i2 * Ss[2] - Pp[2] + k2"),
    ("stride_dropped", "i2 * Ss[2] - Pp[2] + k2 * Dd[2]", "i2 - Pp[2] + k2 * Dd[2]"),
    ("hswish_scale", "const double hs = t * c / 6.0;", "const double hs = t * c / 3.0;"),
    ("hswish_clamp", "if (c > 6.0) c = 6.0;", "if (c > 3.0) c = 3.0;"),
    ("output_padding_ignored", "Lo[e] = ora_out_len(L_in[d], K[d], S[d], P[d], OP[d], DL[d]);",
     "Lo[e] = ora_out_len(L_in[d], K[d], S[d], P[d], 0, DL[d]);"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor for %s not found" % name
    mutated = src.replace(old, new)
    cpath = tmp_path / ("oracle_%s.c" % name)
    cpath.write_text(mutated)
    so = ora.oracle.build_oracle(src=str(cpath), out=str(tmp_path / ("lib_%s.so" % name)), force=True)
    lib = ora.oracle.load_library(so)
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except Exception:  # any failure of a pin counts as "caught"
            failed.append(pin.__name__)
    assert failed, "planted mistake %s passed every pin" % name

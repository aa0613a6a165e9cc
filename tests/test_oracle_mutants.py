"""Plants plausible mistakes in a copy of the oracle's C source and checks that
at least one pin catches each one (so the pins are not vacuous)."""
import os

import pytest

import oracle
from tests.oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "qmv_oracle.c")

# (name, text in the source, replacement)
MUTANTS = [
    ("nibble_order_swapped", "((k & 1) * 4)", "((~k & 1) * 4)"),
    ("offset_7_not_8", "part += (double)(orc_nibble(row, k) - 8) * (double)xt[k];",
     "part += (double)(orc_nibble(row, k) - 7) * (double)xt[k];"),
    ("first_group_scale_only", "acc += (double)s[i * G + g] * part;", "acc += (double)s[i * G] * part;"),
    ("scale_index_transposed", "return (double)(orc_nibble(row, k) - 8) * (double)s[i * (int64_t)(K / gs) + k / gs];",
     "return (double)(orc_nibble(row, k) - 8) * (double)s[(k / gs) * (int64_t)(K / gs) + i % (K / gs)];"),
    ("tie_goes_to_higher_index", "if (best < 0 || orc_route_val(l[e]) > orc_route_val(l[best])) best = e;",
     "if (best < 0 || orc_route_val(l[e]) >= orc_route_val(l[best])) best = e;"),
    ("nan_not_minus_inf", "{ return v != v ? -INFINITY : (double)v; }", "{ return (double)v; }"),
    ("no_renormalisation", "w[(int64_t)t * k + j] = p[ids[(int64_t)t * k + j]] / psum;",
     "w[(int64_t)t * k + j] = p[ids[(int64_t)t * k + j]];"),
    ("silu_sign", "double sg = 1.0 / (1.0 + exp(-g));", "double sg = 1.0 / (1.0 + exp(g));"),
    ("gate_up_swapped", "const uint8_t *urow = gu_q + e * gq_e + (I + c) * (H / 2);",
     "const uint8_t *urow = gu_q + e * gq_e + c * (H / 2);"),
    ("combine_weight_dropped", "o += (double)w[p] * y;", "o += y;"),
    ("group_order_reversed", "for (int64_t p = 0; p < P; ++p) list[fill[ids[p]]++] = (int32_t)p;",
     "for (int64_t p = P - 1; p >= 0; --p) list[fill[ids[p]]++] = (int32_t)p;"),
    ("int8_row_scale_dropped", "y[t * N + i] = (double)r[i] * acc;", "y[t * N + i] = acc;"),
    ("int3_high_bit_msb_first", "const int hi = (g[16 + e / 8] >> (e % 8)) & 1;",
     "const int hi = (g[16 + e / 8] >> (7 - e % 8)) & 1;"),
    ("int3_offset_3_not_4", "const double v = (double)(orc_code3(row, k) - 4);",
     "const double v = (double)(orc_code3(row, k) - 3);"),
    ("moe_den_weight_dropped", "a += fabs((double)w[p]) * ad;", "a += ad;"),
    ("int3_den_scale_dropped", "a += fabs(v * sc * (double)xt[k]);", "a += fabs(v * (double)xt[k]);"),
    ("hden_term_dropped", "hden[p * I + c] = fabs(dsilu * u) * dg + fabs(silu) * du;",
     "hden[p * I + c] = fabs(dsilu * u) * dg;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mpath = tmp_path / f"mut_{name}.c"
    mpath.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(force=True, src=str(mpath), out=str(tmp_path / f"mut_{name}.so")))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"

"""The CPU oracle, pinned to things other than itself (CPU only).

1. Every pin in ``oracle_pins.ALL_PINS`` passes on the oracle as built.
2. Planted mistakes: a copy of the oracle's C source with one plausible bug
   (a dropped term, a wrong sign, a wrong index, a rounding-rule slip, a lost
   carry, ...) is compiled on the CPU and must fail at least one pin.  This is
   what shows the pins can tell a right oracle from a wrong one.
"""
from __future__ import annotations

import os

import pytest

import oracle
import oracle_pins


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda p: p.__name__)
def test_pin(orc, pin):
    pin(orc)


# (name, [(text in skinny_oracle.c, replacement), ...])
MUTANTS = [
    ("drop_last_term",
     [("for (k = 0; k < j->K; ++k) {", "for (k = 0; k < j->K - 1; ++k) {"),
      ("for (k = 0; k < K; ++k) {\n        bf16_parts xp", "for (k = 0; k < K - 1; ++k) {\n        bf16_parts xp")]),
    ("truncate_instead_of_round",
     [("if (round && (sticky || (q & 1u))) q += 1;", "if (0) q += 1;")]),
    ("ties_away_from_zero",
     [("if (round && (sticky || (q & 1u))) q += 1;", "if (round) q += 1;")]),
    ("ties_to_odd",
     [("if (round && (sticky || (q & 1u))) q += 1;", "if (round && (sticky || !(q & 1u))) q += 1;")]),
    ("sticky_bits_ignored",
     [("for (i = ql - 2; i >= 0 && !sticky; --i) sticky = acc_bit(a, i);", "")]),
    ("sign_of_x_only",
     [("int neg = x->neg ^ w->neg;", "int neg = x->neg;")]),
    ("shifted_w_index",
     [("bf16_parts wp = decode_bf16(wrow[k]);", "bf16_parts wp = decode_bf16(wrow[(k + 1) % j->K]);"),
      ("bf16_parts xp = decode_bf16(x[k]), wp = decode_bf16(w[k]);",
       "bf16_parts xp = decode_bf16(x[k]), wp = decode_bf16(w[(k + 1) % K]);")]),
    ("always_row_zero_of_x",
     [("const bf16_parts *xr = j->xp + (long long)m * j->K;", "const bf16_parts *xr = j->xp;")]),
    ("subnormal_exponent_off_by_one",
     [("p.pos = 0;          /* e = -133 */", "p.pos = 1;          /* e = -133 */")]),
    ("lost_high_digit",
     [("a->d[i + 1] += hi;", "(void)hi;")]),
    ("no_overflow_to_inf",
     [("if (u > 120) return (uint16_t)(s | 0x7f80);", "")]),
    ("inf_times_zero_not_nan",
     [("if (other == 0)\n            a->nan = 1;", "if (0)\n            a->nan = 1;")]),
    ("f32_one_bit_short",
     [("acc_round(a, 24, -149, &q, &u);", "acc_round(a, 23, -149, &q, &u);")]),
    ("f32_exponent_bias_off_by_one",
     [("return s | ((uint32_t)(u + 150) << 23)", "return s | ((uint32_t)(u + 151) << 23)")]),
    ("f32_no_overflow_to_inf",
     [("if (u > 104) return s | 0x7f800000u;", "")]),
    ("f32_flush_subnormals",
     [("if (q < ((uint64_t)1 << 23)) return s | (uint32_t)q;", "if (q < ((uint64_t)1 << 23)) return s;")]),
    ("f32_rounded_through_bf16",
     [("j->y32[(long long)m * j->ldy + n] = acc_to_f32(&acc);",
       "j->y32[(long long)m * j->ldy + n] = (uint32_t)acc_to_bf16(&acc) << 16;")]),
]


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, edits):
    src = open(oracle.SOURCE).read()
    for old, new in edits:
        assert old in src, f"mutation {name}: text not found in the oracle source"
        src = src.replace(old, new)
    path = tmp_path / f"mutant_{name}.c"
    path.write_text(src)
    lib = oracle.compile_library(str(path), str(tmp_path / f"libmutant_{name}.so"))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name!r} passed every pin"
    os.remove(lib)

"""Planted mistakes: each mutant is a copy of the oracle source with one
plausible error (a dropped term, a wrong sign, index or constant, another
rounding).  It is compiled on the CPU into a temporary library, and the pins in
test_oracle_codecs.py / test_oracle_ops.py must reject it."""
import os
import subprocess

import pytest

import exact_ref as X
import oracle as O
import test_oracle_codecs as C
import test_oracle_ops as P
import test_oracle_rope as RP

SRC = os.path.join(os.path.dirname(O.__file__), "fp8norm_oracle.c")

MUTANTS = {
    "eps_dropped": ("float v = ms + eps;", "float v = ms;"),
    "mean_square_exponent_off_by_one": ("return (float)ldexp((double)mant, shift - 330);",
                                        "return (float)ldexp((double)mant, shift - 331);"),
    "sigmoid_sign_flipped": ("double sig = 1.0 / (1.0 + exp(-x));",
                             "double sig = 1.0 / (1.0 + exp(x));"),
    "fp8_max_240": ("float scale = famax / 448.0f;", "float scale = famax / 240.0f;"),
    "normalised_value_not_rounded": (
        "return oracle_bf16_from_double(oracle_bf16_to_double(xnb) * oracle_bf16_to_double(wb));",
        "return oracle_bf16_from_double((double)xn * oracle_bf16_to_double(wb));"),
    "weight_reversed": ("uint16_t u = norm_times_weight(xh[d], r, weight[d]);",
                        "uint16_t u = norm_times_weight(xh[d], r, weight[D - 1 - d]);"),
    "mx_emax_7": ("int e = (e2 - 1) - 8;", "int e = (e2 - 1) - 7;"),
    "e4m3_ties_away": ("int qexp = (E < -6) ? -9 : E - 3; /* quantum of the binade (or subnormal) */\n"
                       "  double n = rint(ldexp(a, -qexp));",
                       "int qexp = (E < -6) ? -9 : E - 3;\n  double n = round(ldexp(a, -qexp));"),
    "static_descale_of_wrong_head": ("out[(t * H + h) * Dh + d] = oracle_e4m3_from_float(xv / descale[h]);",
                                     "out[(t * H + h) * Dh + d] = oracle_e4m3_from_float(xv / descale[H - 1 - h]);"),
    "static_multiplies": ("out[(t * H + h) * Dh + d] = oracle_e4m3_from_float(xv / descale[h]);",
                          "out[(t * H + h) * Dh + d] = oracle_e4m3_from_float(xv * (1.0f / descale[h]));"),
    "inv_rope_forward_rotation": ("float y1 = a + b;", "float y1 = a - b;"),
    "inv_rope_pairs_swapped": ("int32_t j1 = interleaved ? rope_off + 2 * i : rope_off + i;",
                               "int32_t j1 = !interleaved ? rope_off + 2 * i : rope_off + i;"),
    "bf16_truncates": ("double n = rint(ldexp(a, -qexp)); /* ties to even (default rounding mode) */",
                       "double n = floor(ldexp(a, -qexp));"),
}


def _pins(act_tabs):
    return [
        C.test_bf16_from_binary32_matches_torch_cast,
        C.test_e4m3_ties_saturation_and_specials,
        C.test_e4m3_roundtrip_all_codes,
        lambda: C.test_activation_exhaustive_against_decimal(O.ACT_SIGMOID, "sigmoid"),
        lambda: C.test_mean_square_matches_exact(40),
        C.test_rms_factor_matches_exact,
        C.test_e8m0_code_all_positive_bf16,
        P.test_golden_gated_unit_rows,
        P.test_golden_mx_unit_rows,
        P.test_golden_static_unit_rows,
        lambda: P.test_gated_matches_exact_checker(2, 1, 128, "silu", act_tabs),
        lambda: P.test_static_matches_exact_checker(3, 2, 24),
        lambda: P.test_mx_matches_exact_checker(2, 64, 40),
        RP.test_golden_inv_rope_rows,
        lambda: RP.test_inv_rope_matches_exact_checker(2, 64, 32, 32, True),
    ]


@pytest.fixture(scope="module")
def act_tabs():
    return {"sigmoid": X.act_table_exact("sigmoid"), "silu": X.act_table_exact("silu")}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, act_tabs, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: " + name
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    inc = os.path.dirname(SRC)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-I", inc,
                    str(mpath), "-o", str(lib), "-lm"], check=True)
    real = O.lib()
    O.use_library(O.load_library(str(lib)))
    caught = []
    try:
        for pin in _pins(act_tabs):
            try:
                pin()
            except AssertionError:
                caught.append(getattr(pin, "__name__", "pin"))
    finally:
        O.use_library(real)
    assert caught, "no pin rejected the mutant " + name

"""The oracle's pins must catch plausible mistakes.  Each case plants one
mistake in a copy of the oracle's C source (on the CPU), compiles it, swaps it
in for the real oracle and checks that at least one pin test fails."""
import ctypes
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    # bias subtracted instead of added (the bug rlx-moshi's doc comment names)
    "bias_subtracted": ("return fmaf(s, (float)code, b);", "return fmaf(s, (float)code, -b);"),
    # bias dropped
    "bias_dropped": ("return fmaf(s, (float)code, b);", "return fmaf(s, (float)code, 0.0f);"),
    # fp16 output truncated instead of rounded to nearest even
    "f16_truncation": ("double r = nearbyint(a / q) * q;", "double r = floor(a / q) * q;"),
    # fp16 exponent bias off by one
    "f16_exponent_bias": ("v = ldexp((double)(1024 + f), e - 25);",
                          "v = ldexp((double)(1024 + f), e - 24);"),
    # fp16 subnormals read with the normal numbers' implicit one
    "f16_subnormal": ("v = ldexp((double)f, -24);", "v = ldexp((double)(1024 + f), -24);"),
    # typed matmul reads x as bf16 whatever its type
    "x_type_ignored": ("double t = load_elem(c->x, c->x_type, m * c->K + k) * w[k];",
                       "double t = load_elem(c->x, ORACLE_BF16, m * c->K + k) * w[k];"),
    # most significant bit first inside a code
    "msb_first": ("code |= stream_bit(row_words, j * (int64_t)bits + t) << t;",
                  "code |= stream_bit(row_words, j * (int64_t)bits + t) << (bits - 1 - t);"),
    # group index along the wrong position (one group per code)
    "wrong_group": ("int64_t g = j / c->group_size;", "int64_t g = (j / c->group_size + 1) % groups;"),
    # fp64 matmul weight with transposed stored index
    "transposed_operand": ("int64_t row = transpose ? n : k;", "int64_t row = transpose ? k : n;"),
    # bf16 output truncated instead of rounded to nearest even
    "bf16_truncation": ("u += 0x7FFFu + kept_lsb;", "u += 0u * kept_lsb;"),
    # matmul weight uses the bias twice
    "matmul_bias_twice": ("return s * (double)code + b;", "return s * (double)code + 2.0 * b;"),
}

PIN_TESTS = [
    (pins.test_lsb_first_plus_bias, ()),
    (pins.test_identity_shape, ()),
    (pins.test_int8_byte_layout, ()),
    (pins.test_three_bit_stream_by_hand, ()),
    (pins.test_constant_weight_matmul, ()),
    (pins.test_unpack_matches_numpy_unpackbits, (3,)),
    (pins.test_zero_codes_give_bias, (4,)),
    (pins.test_dequant_f32_is_exact_value_rounded_once, (4, 64)),
    (pins.test_bf16_rounding_matches_torch, ()),
    (pins.test_dequant_bf16_is_rne_of_f32, (4,)),
    (pins.test_qmm_brute_force_tiny, (4, 64, True)),
    (pins.test_qmm_brute_force_tiny, (4, 64, False)),
    (pins.test_transpose_flag_is_not_a_no_op, ()),
    (pins.test_rows_is_a_gather_of_dequantize, ()),
    (pins.test_f16_to_f64_matches_numpy_every_pattern, ()),
    (pins.test_f32_to_f16_matches_numpy, ()),
    (pins.test_typed_dequant_pins, ("f16",)),
    (pins.test_typed_dequant_pins, ("f32",)),
    (pins.test_typed_dequant_f16_out_is_rne_of_f32, ("f32",)),
    (pins.test_typed_qmm_brute_force_tiny, ("f16", "f16", True)),
    (pins.test_typed_qmm_brute_force_tiny, ("f32", "bf16", False)),
]


def _build_mutant(tmp_path, old, new):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "qmm_oracle.c")).read()
    assert src.count(old) == 1, old
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=gnu99", "-O1", "-ffp-contract=off", "-fPIC", "-shared",
                    "-pthread", str(path), "-o", str(lib), "-lm"], check=True)
    return str(lib)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path, monkeypatch):
    real = oracle._load()
    mutant = ctypes.CDLL(_build_mutant(tmp_path, *MUTANTS[name]))
    # Give the mutant the same prototypes as the real library.
    for sym in ("oracle_code", "oracle_unpack", "oracle_pack", "oracle_bf16_to_f32",
                "oracle_f32_to_bf16", "oracle_dequantize", "oracle_rows", "oracle_qmm",
                "oracle_qmm_sampled", "oracle_quantize", "oracle_f16_to_f64",
                "oracle_f32_to_f16", "oracle_dequantize_typed", "oracle_rows_typed",
                "oracle_qmm_typed", "oracle_qmm_sampled_typed", "oracle_quantize_typed"):
        f, g = getattr(real, sym), getattr(mutant, sym)
        g.argtypes, g.restype = f.argtypes, f.restype
    monkeypatch.setattr(oracle, "_lib", mutant)
    caught = []
    for test, args in PIN_TESTS:
        try:
            test(*args)
        except AssertionError:
            caught.append(test.__name__)
    assert caught, "no pin caught the planted mistake %r" % name

"""Plants plausible mistakes in copies of the oracle's C source, on the CPU,
and checks that the pin suite rejects every one of them: evidence that the
pins would catch a dropped term, a wrong sign, index, shift or field offset.
"""
import os

import numpy as np

import pytest

import oracle
import oracle_pins as P

MUTANTS = {
    # Figure 6.1 geometry
    "q6_block_bytes": ("case KQO_Q6_K: return 210;", "case KQO_Q6_K: return 208;"),
    # binary16 decode
    "f16_exponent_bias": ("e - 25);", "e - 24);"),
    "f16_subnormal": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    # 6-bit scale / min unpacking (Figure 6.3)
    "scale_low_wrong_byte": ("*m = scales[j + 4] & 63;", "*m = scales[j] & 63;"),
    "scale_hi_wrong_source": ("((scales[j - 4] >> 6) << 4)", "((scales[j] >> 6) << 4)"),
    "min_hi_dropped": ("*m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);",
                       "*m = (scales[j + 4] >> 4);"),
    # Q4_K / Q5_K element map and formula
    "min_sign": ("out[64 * g + l] = d_lo * (float)code_lo - min_lo;",
                 "out[64 * g + l] = d_lo * (float)code_lo + min_lo;"),
    "nibble_interleave": ("out[64 * g + 32 + l]", "out[64 * g + 16 + l]"),
    "hi_uses_lo_scale": ("const float d_hi = d * (float)sc_hi",
                         "const float d_hi = d * (float)sc_lo"),
    "q5_qh_bit": ("((qh[l] >> (2 * g)) & 1) << 4", "((qh[l] >> (2 * g + 1)) & 1) << 4"),
    "q5_qs_offset": ("b + (has_qh ? 48 : 16)", "b + (has_qh ? 16 : 16)"),
    "dmin_offset": ("le16(b + 2)", "le16(b + 0)"),
    # Q6_K
    "q6_offset_32": ("out[idx] = scale * (float)(code[k] - 32);",
                     "out[idx] = scale * (float)(code[k] - 31);"),
    "q6_scale_index": ("sc[idx / 16]", "sc[idx / 32]"),
    "q6_d_offset": ("le16(b + 208)", "le16(b + 206)"),
    "q6_quadrant_swap": ("code[1] = (L[l + 32] & 15)", "code[1] = (L[l] & 15)"),
    "q6_qh_shift": ("(((H[l] >> 4) & 3) << 4)", "(((H[l] >> 6) & 3) << 4)"),
    # matvec
    "f32_accumulation": ("acc += p;", "acc = (double)(float)(acc + p);"),
    "magnitude_signed": ("mag += fabs(p);", "mag += p;"),
    "row_stride": ("const uint8_t *r = W + row * nb * bb;",
                   "const uint8_t *r = W + row * bb;"),
    "transposed_dense": ("dot_f64(W + i * cols, x + t * cols",
                         "dot_f64(W + t * cols, x + i * cols"),
}


def _run_all(o):
    failed = []
    for pin in P.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(os.path.join(os.path.dirname(oracle.__file__),
                            "kq_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    path = tmp_path / "kq_oracle_mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_library(str(path), str(tmp_path / "libmut.so"))
    # a mutant may produce non-finite weights; numpy's notes about them are
    # beside the point, the pins' verdict is what counts
    with np.errstate(all="ignore"):
        failed = _run_all(oracle.Oracle(lib))
    assert failed, f"mutant {name} passed every pin"

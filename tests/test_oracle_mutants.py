"""Planted mistakes in the oracle must fail at least one pin.

Each mutant is a one-line textual change to a temporary copy of
``oracle/kamera_oracle.c`` (a flipped sign, a wrong pair index, a wrong
frequency, a transposed or swapped factor, a dropped term, a wrong rounding
step, a lost offset).  It is built with gcc into a temporary directory, loaded
and run through the whole pin battery on the CPU.  The mutant passes the test
only by failing a pin; a mutant that every pin accepts would be a mistake the
oracle could carry unnoticed.
"""
import os
import tempfile

import pytest

import oracle as O
from tests import oracle_pins as P

MUTANTS = {
    "rotation_sign_a": ("x[a] = xa * c - xb * s;", "x[a] = xa * c + xb * s;"),
    "rotation_sign_b": ("x[b] = xb * c + xa * s;", "x[b] = xb * c - xa * s;"),
    "delta_sign": ("double phi = (double)delta * inv_freq[i];",
                   "double phi = -(double)delta * inv_freq[i];"),
    "rotate_half_partner": ("*b = rot_offset + i + rot_dim / 2;",
                            "*b = rot_offset + rot_dim - 1 - i;"),
    "interleaved_pair": ("*a = rot_offset + 2 * i;\n        *b = rot_offset + 2 * i + 1;",
                         "*a = rot_offset + i;\n        *b = rot_offset + i + rot_dim / 2;"),
    "theta_exponent": ("pow(base, -2.0 * (double)i / (double)rot_dim)",
                       "pow(base, -1.0 * (double)i / (double)rot_dim)"),
    "theta_index": ("pow(base, -2.0 * (double)i / (double)rot_dim)",
                    "pow(base, -2.0 * (double)(i + 1) / (double)rot_dim)"),
    "zero_delta_not_identity": ("    if (delta == 0)\n        return;\n    for (int i = 0; i < rot_dim / 2; ++i) {",
                                "    for (int i = 0; i < rot_dim / 2; ++i) {"),
    "vm_transposed": ("vm[(size_t)c * m + r]", "vm[(size_t)r * width + c]"),
    "patch_dropped": ("y[c] += acc;", "y[c] += 0.0 * acc;"),
    "round_half_up": ("double n = rint(a / q);", "double n = floor(a / q + 0.5);"),
    "round_truncate": ("double n = rint(a / q);", "double n = trunc(a / q);"),
    "bf16_mantissa_width": ("double q = ldexp(1.0, e - 7);", "double q = ldexp(1.0, e - 8);"),
    "bf16_subnormal_floor": ("if (e < -126)\n        e = -126;", "if (e < -120)\n        e = -120;"),
    "gqa_k_uses_value_factor": ("uk = p0[c] + (lh * T + j) * m;", "uk = p2[c] + (lh * T + j) * m;"),
    "gqa_vm_layer_dropped": ("vk = p1[c] + lh * (int64_t)d * m;",
                             "vk = p1[c] + (int64_t)h * d * m;"),
    "gqa_head_offset_dropped": ("const int64_t so = l * store_layer_stride + src * store_row_stride + (int64_t)h * d;",
                                "const int64_t so = l * store_layer_stride + src * store_row_stride;"),
    "gqa_src_offset_dropped": ("const int64_t src = src_offset[c] + j;", "const int64_t src = j;"),
    "gqa_values_rotated": ("kamera_oracle_row(store_v + so, d, 0, 0,",
                           "kamera_oracle_row(store_v + so, d, 1, delta[c],"),
    "mla_rope_not_rotated": ("kamera_oracle_row(store + so + kv_lora, rope_dim, 1, delta[c],",
                             "kamera_oracle_row(store + so + kv_lora, rope_dim, 0, delta[c],"),
    "mla_rope_factor_swapped": ("ur = p2[c] + ((int64_t)l * T + j) * m;",
                                "ur = p0[c] + ((int64_t)l * T + j) * m;"),
    "ingest_row_offset_dropped": ("const int64_t so = l * store_layer_stride + (dst_row[c] + j) * store_row_stride;",
                                  "const int64_t so = l * store_layer_stride + (int64_t)j * store_row_stride;"),
    "ingest_values_not_copied": ("if (pool_v)\n                    memcpy(", "if (0)\n                    memcpy("),
    "slide_offset_ignored": ("kamera_oracle_row(row, d, 1, delta[c], inv_freq, rot_dim, rot_offset, pairing,",
                             "kamera_oracle_row(row, d, 1, delta[c], inv_freq, rot_dim, 0, pairing,"),
}


@pytest.fixture(scope="module")
def source():
    with open(O.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) == 1, f"mutation site for {name} not unique/present"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = O.build(str(tmp_path / "libmutant.so"), source=str(src))
    orc = O.Oracle(lib)
    caught = []
    for pin in P.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"

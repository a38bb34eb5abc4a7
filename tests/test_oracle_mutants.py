"""Negative controls: plant a plausible mistake in a copy of the oracle's C
source, build it, and require that the pins catch it.  A pin set that never
goes red proves nothing."""
import os
import shutil

import pytest

import oracle
from _pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "iq4xs_oracle.c")

# (name, text in the real source, planted replacement)
MUTANTS = [
    ("swap_nibble_halves",
     "int nib = (i < 16) ? (byte & 0x0F) : (byte >> 4);\n    return or_kvalues[nib];",
     "int nib = (i < 16) ? (byte >> 4) : (byte & 0x0F);\n    return or_kvalues[nib];"),
    ("ls_minus_31", "(float)(oracle_iq4xs_ls(block, j) - 32)", "(float)(oracle_iq4xs_ls(block, j) - 31)"),
    ("scales_l_nibble_order",
     "int lo = (j & 1) ? (scales_l[j / 2] >> 4) : (scales_l[j / 2] & 0x0F);",
     "int lo = (j & 1) ? (scales_l[j / 2] & 0x0F) : (scales_l[j / 2] >> 4);"),
    ("scales_h_reversed", "int hi = (scales_h >> (2 * j)) & 3;", "int hi = (scales_h >> (2 * (7 - j))) & 3;"),
    ("codebook_typo", "-127, -104, -83, -65", "-127, -104, -82, -65"),
    ("round_half_even", "q = (int)roundf(t);", "q = (int)rintf(t);"),
    ("d_over_128", "float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    ("s_without_d", "oracle_f32_to_f16(d * (float)sum)", "oracle_f32_to_f16((float)sum)"),
    ("drop_activation_scale", "acc += sw * dx * (double)P;\n                }",
     "acc += sw * (double)P;\n                }"),
    ("qs_byte_offset", "uint8_t byte = block[OR_OFF_QS + 16 * j + (i % 16)];",
     "uint8_t byte = block[OR_OFF_QS + 16 * j + (i % 16) + (i >= 16)];"),
    ("f16_tie_rounds_up", "if (r < 0.5) return fl;", "if (r < 0.5) return fl;\n    return fl + 1.0;"),
    ("f16_subnormal_scale", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    ("q4_0_minus_7", "? nib - 8 : or_kvalues[nib];", "? nib - 7 : or_kvalues[nib];"),
    ("b18_formats_swapped", "return (wtype == OR_WT_Q4_0) ? nib - 8", "return (wtype != OR_WT_Q4_0) ? nib - 8"),
    ("b18_nibble_halves", "int nib = (i < 16) ? (byte & 0x0F) : (byte >> 4);\n    return (wtype",
     "int nib = (i < 16) ? (byte >> 4) : (byte & 0x0F);\n    return (wtype"),
    ("b18_qs_offset", "#define OR_B18_OFF_QS 2", "#define OR_B18_OFF_QS 1"),
    ("b18_scale_bytes", "(uint16_t)(block[0] | (block[1] << 8))", "(uint16_t)(block[1] | (block[0] << 8))"),
    ("b18_block_stride", "c * OR_B18_BYTES, i);", "c * 16, i);"),
    ("wt_drop_activation_scale", "acc += sw * dx * (double)P;\n            }\n            job->y[m * job->N + n] = acc;\n        }\n    }\n    return NULL;\n}\n\n/* y[M][N] (double) for weights",
     "acc += sw * (double)P;\n            }\n            job->y[m * job->N + n] = acc;\n        }\n    }\n    return NULL;\n}\n\n/* y[M][N] (double) for weights"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path, kvalues):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site for {name} not found exactly once"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new))
    lib_path = oracle.compile_oracle(str(src), str(tmp_path / "libmutant.so"))
    orc = oracle.Oracle(oracle.load_library(lib_path))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(orc, kvalues)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"

"""Mutation check of the oracle's pins (no GPU).

Each mutant below is one plausible slip in the oracle's C source (a flipped bit order,
a dropped term, a wrong field, a missing check). The test compiles the mutated copy in
a temporary directory and runs the oracle's pin suite against it in a subprocess; the
suite must fail for every mutant. The committed oracle itself is never modified.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "bit_order": ("mask |= 1u << i;", "mask |= 1u << (31u - i);"),
    "zero_test_ignores_sign": ("x[w0 + i] != 0u", "(x[w0 + i] & 0x7fffffffu) != 0u"),
    "value_bits": ("put_u32(payload + cur, x[w0 + i]);", "put_u32(payload + cur, x[w0 + i] ^ 1u);"),
    "chunk_offset_off_by_word": ("put_u64(out + ZVCO_STREAM_HEADER_BYTES + 8 * c, cur);",
                                 "put_u64(out + ZVCO_STREAM_HEADER_BYTES + 8 * c, cur + 4 * (c > 0));"),
    "table_entry_width": ("const uint64_t payload_start = ZVCO_STREAM_HEADER_BYTES + 8 * nc;\n  if (cap",
                          "const uint64_t payload_start = ZVCO_STREAM_HEADER_BYTES + 4 * nc;\n  if (cap"),
    "word_bytes_field": ("put_u16(out + 6, 4);", "put_u16(out + 6, 32);"),
    "payload_field_absolute": ("put_u64(out + 24, cur);", "put_u64(out + 24, payload_start + cur);"),
    "decode_no_zero_fill": ("y[w0 + i] = 0u;", "(void)y;"),
    "decode_no_end_check": ("if (cur != end) return ZVCO_ERR_CORRUPT;", "(void)end;"),
    "decode_no_tail_check": ("if (valid < ZVCO_WINDOW && (mask >> valid) != 0u) return ZVCO_ERR_CORRUPT;",
                             "(void)valid;"),
    "decode_mask_popcount": ("cur += 4;\n      const uint64_t valid", "cur += 8;\n      const uint64_t valid"),
    "batch_last_offset": ("put_u64(out + ZVCO_BATCH_HEADER_BYTES + 8 * (uint64_t)T, pos);",
                          "put_u64(out + ZVCO_BATCH_HEADER_BYTES + 8 * (uint64_t)T, pos - 4);"),
    "batch_magic": ("put_u32(out + 0, ZVCO_BATCH_MAGIC);", "put_u32(out + 0, ZVCO_STREAM_MAGIC);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "zvc_oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut_src = tmp_path / "zvc_oracle_mutant.c"
    mut_src.write_text(src.replace(old, new))
    lib = oracle.build(str(mut_src), str(tmp_path / "libmutant.so"),
                       extra_flags=("-Wno-unused-variable", "-Wno-unused-but-set-variable"))
    env = dict(os.environ, ZVC_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the oracle pins:\n{r.stdout[-2000:]}"


# The 16-bit oracle (zvc16_oracle.c) against its own pin suite.
MUTANTS16 = {
    "bit_order": ("if (x[w + i] != 0) mask |= 1u << i;", "if (x[w + i] != 0) mask |= 1u << (31u - i);"),
    "zero_test_ignores_sign": ("if (x[w + i] != 0) mask", "if ((x[w + i] & 0x7fffu) != 0) mask"),
    "zero_test_low_byte": ("if (x[w + i] != 0) mask", "if ((x[w + i] & 0xffu) != 0) mask"),
    "value_byte_order": ("wr8(out + start + at, x[w + i], ZVCO16_WORD_BYTES);",
                         "wr8(out + start + at, (uint16_t)((x[w + i] >> 8) | (x[w + i] << 8)), "
                         "ZVCO16_WORD_BYTES);"),
    "values_padded_to_words": ("wr8(out + start + at, x[w + i], ZVCO16_WORD_BYTES);\n"
                               "        at += ZVCO16_WORD_BYTES;",
                               "wr8(out + start + at, x[w + i], ZVCO16_WORD_BYTES);\n"
                               "        at += 4;"),
    "mask_two_bytes": ("wr8(out + start + at, mask, 4);\n      at += 4;",
                       "wr8(out + start + at, mask, 2);\n      at += 2;"),
    "word_bytes_field": ("wr8(out + 6, ZVCO16_WORD_BYTES, 2);", "wr8(out + 6, 4, 2);"),
    "chunk_offset_off_by_two": ("wr8(out + ZVCO16_HEADER_BYTES + 8 * c, at, 8);",
                                "wr8(out + ZVCO16_HEADER_BYTES + 8 * c, at + 2 * (c > 0), 8);"),
    "decode_no_zero_fill": ("y[w + i] = 0;", "(void)y;"),
    "decode_no_end_check": ("if (at != stop) return ZVCO16_ERR_CORRUPT;", "(void)stop;"),
    "decode_no_tail_check": ("if (count < ZVCO16_WINDOW && (mask >> count) != 0u) return ZVCO16_ERR_CORRUPT;",
                             "(void)count;"),
    "decode_reads_high_byte_only": ("y[w + i] = (uint16_t)rd8(in + start + at, ZVCO16_WORD_BYTES);",
                                    "y[w + i] = (uint16_t)(rd8(in + start + at + 1, 1) << 8);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS16))
def test_pins_catch_mutant16(name, tmp_path):
    old, new = MUTANTS16[name]
    src = open(os.path.join(ROOT, "oracle", "zvc16_oracle.c")).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mut_src = tmp_path / "zvc16_oracle_mutant.c"
    mut_src.write_text(src.replace(old, new))
    lib = oracle.build(str(mut_src), str(tmp_path / "libmutant16.so"),
                       extra_flags=("-Wno-unused-variable", "-Wno-unused-but-set-variable"))
    env = dict(os.environ, ZVC16_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_zvc16_oracle.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the 16-bit oracle pins:\n{r.stdout[-2000:]}"

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

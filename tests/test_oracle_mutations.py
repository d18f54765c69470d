"""Pin strength: plant plausible mistakes in a copy of the oracle's C source and
check that at least one pin of test_oracle_pins.py fails for each.

Each mutation is a textual edit (of the first match) in oracle/splitzip_oracle.c compiled into a
temporary library; the real oracle is untouched.  A mutation whose target text
is missing fails the test, so edits to the oracle keep this list honest.
"""
import pytest

import oracle
from tests import test_oracle_pins as pins
from tests.golden_io import STREAM_FIXTURES

MUTATIONS = {
    "exponent_shift": ("return (u >> 7) & 0xFFu;", "return (u >> 8) & 0xFFu;"),
    "nibble_order": ("if (i % 2 == 0)\n        codes[i / 2] = (uint8_t)((codes[i / 2] & 0xF0u) | code);",
                     "if (i % 2 == 1)\n        codes[i / 2] = (uint8_t)((codes[i / 2] & 0xF0u) | code);"),
    "global_position": ("esc_pos[E] = (uint16_t)p;", "esc_pos[E] = (uint16_t)i;"),
    "escape_code_15": ("E++;\n                code = 0;", "E++;\n                code = 15;"),
    "tie_to_larger": ("hist[b] > hist[best]", "hist[b] >= hist[best]"),
    "signman_swap": ("signman[i] = (uint8_t)((bf16_sign(u) << 7) | bf16_mantissa(u));",
                     "signman[i] = (uint8_t)((bf16_mantissa(u) << 1) | bf16_sign(u));"),
    "e5m2_field_order": ("put_field3(signman, i, (e5m2_sign(u) << 2) | e5m2_mantissa(u));",
                         "put_field3(signman, i, (e5m2_mantissa(u) << 1) | e5m2_sign(u));"),
    "e5m2_exponent_mask": ("return (u >> 2) & 0x1Fu;", "return (u >> 2) & 0x0Fu;"),
    "size_drops_metadata": ("3 * E + 4 * (ceil_div(n, chunk) + 1);\n}\n\nuint64_t oracle_compressed_bytes_e5m2",
                            "3 * E + 4 * ceil_div(n, chunk);\n}\n\nuint64_t oracle_compressed_bytes_e5m2"),
    "decode_skips_patch": ("y[start + p] = bf16_assemble(bf16_sign(u), esc_val[j], bf16_mantissa(u));",
                           "y[start + p] = u;"),
    "decode_sign_from_mantissa_bit": ("y[i] = bf16_assemble((sm >> 7) & 1u, e, sm & 0x7Fu);",
                                      "y[i] = bf16_assemble((sm >> 6) & 1u, e, sm & 0x7Fu);"),
    "chunk_off_inclusive": ("chunk_off[c] = (uint32_t)E;\n        for (uint64_t p = 0; p < len; p++) {\n            uint64_t i = start + p;\n            uint16_t u = x[i];",
                            "chunk_off[c] = (uint32_t)E + (c > 0);\n        for (uint64_t p = 0; p < len; p++) {\n            uint64_t i = start + p;\n            uint16_t u = x[i];"),
}

PIN_CALLS = (
    [lambda n=n: pins.test_golden_encode_streams(n) for n in STREAM_FIXTURES]
    + [lambda n=n: pins.test_golden_decode_streams(n) for n in STREAM_FIXTURES]
    + [pins.test_golden_top16_tie_rule,
       pins.test_all_bf16_patterns_self_calibrated,
       pins.test_all_e5m2_patterns,
       lambda: pins.test_histogram_matches_bincount("e5m2"),
       lambda: pins.test_top16_matches_lexsort(1)]
)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = oracle.source_text()
    assert src.count(old) >= 1, f"mutation target for {name} not found"
    so = oracle.compile_variant(src.replace(old, new, 1), str(tmp_path))
    failures = 0
    with oracle.use_library(so):
        for call in PIN_CALLS:
            try:
                call()
            except Exception:
                failures += 1
    assert failures > 0, f"no pin caught mutation {name}"

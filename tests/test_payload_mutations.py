"""Pin strength for the payload oracle: plant plausible mistakes in a copy of
oracle/payload.py and check that a pin fails for each.

Each mutation is a textual edit (of the first match) loaded as a separate
module inside the oracle package; the real module is untouched.  A mutation
whose target text is missing fails the test, so edits to the payload oracle
keep this list honest.  The pins: the hand-worked payloads of tests/golden/
(exact bytes, slice table, decode), a round trip with one codebook per
slice, and the per-slice calibrated payloads whose codebooks are worked out by
hand in tests/test_payload.py.
"""
import os
import types

import numpy as np
import pytest

import oracle
from tests.golden_io import hex_array, load

SRC = os.path.join(os.path.dirname(oracle.__file__), "payload.py")

MUTATIONS = {
    "dense_regions_unpadded": (
        "            region += bytes(_pad16(len(region)) - len(region))\n        dense.append(",
        "        dense.append("),
    "escape_values_first": (
        'region = (np.asarray(st["esc_pos"], np.uint16).tobytes() +\n'
        '                  np.asarray(st["esc_val"], np.uint8).tobytes())',
        'region = (np.asarray(st["esc_val"], np.uint8).tobytes() +\n'
        '                  np.asarray(st["esc_pos"], np.uint16).tobytes())'),
    "escapes_before_dense": ("for region in dense + escapes:", "for region in escapes + dense:"),
    "entry_offsets_swapped": ("ENTRY.pack(m, e, d, q, bytes(cb))", "ENTRY.pack(m, e, q, d, bytes(cb))"),
    "format_codes_swapped": ('FORMAT_CODE = {"bf16": 0, "e5m2": 1}', 'FORMAT_CODE = {"bf16": 1, "e5m2": 0}'),
    "header_counts_first_slice": ("chunk, sum(n_esc), total)", "chunk, n_esc[0], total)"),
    "first_codebook_for_all": ("ENTRY.pack(m, e, d, q, bytes(cb))", "ENTRY.pack(m, e, d, q, bytes(cbs[0]))"),
    "reader_chunk_off_unaligned": ("        p = _pad16(p + n_sm)\n", "        p = p + n_sm\n"),
    "calibrated_on_whole_tensor": ("_calibrate(x[s0:s0 + m], fmt)", "_calibrate(x, fmt)"),
    "calibrated_on_first_slice": ("_calibrate(x[s0:s0 + m], fmt)", "_calibrate(x[:m], fmt)"),
    "calibrated_slice_cut_short": ("_calibrate(x[s0:s0 + m], fmt)", "_calibrate(x[s0:s0 + m - 16], fmt)"),
}

FIXTURES = ["payload_bf16_two_slices.txt", "payload_e5m2_two_slices.txt"]


def _variant(src: str) -> types.ModuleType:
    mod = types.ModuleType("oracle._payload_variant")
    mod.__package__ = "oracle"
    exec(compile(src, "payload_variant.py", "exec"), mod.__dict__)
    return mod


def _pin_fixture(op, name):
    fx = load(name)
    fmt = fx["format"][0]
    rows = sorted((int(k.split("@")[1]), v) for k, v in fx.items() if k.startswith("payload@"))
    ref = bytes(int(t, 16) for _, v in rows for t in v)
    x = hex_array(fx["input_hex"], np.uint16 if fmt == "bf16" else np.uint8)
    cb = [int(c) for c in fx["codebook"]]
    chunk, se = int(fx["chunk"][0]), int(fx["slice_elems"][0])
    assert op.write(x, fmt, chunk, se, cb) == ref
    head, slices = op.read(ref)
    assert head["fmt"] == fmt and head["n_escapes"] == int(fx["n_escapes"][0])
    assert [s["off_dense"] for s in slices] == [int(v) for v in fx["slice_off_dense"]]
    assert [s["off_escapes"] for s in slices] == [int(v) for v in fx["slice_off_escapes"]]
    assert np.array_equal(op.decode(ref), x)


def _pin_per_slice_codebooks(op):
    rng = np.random.default_rng(3)
    a = (rng.standard_normal(3000).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    b = (a & 0x807F) | (100 << 7)   # a second slice whose exponents are all 100
    x = np.concatenate([a, b])
    cbs = [[int(c) for c in oracle.calibrate(part, "bf16")[0]] for part in (x[:3072], x[3072:])]
    buf = op.write(x, "bf16", 256, 3072, cbs)
    _, slices = op.read(buf)
    assert [s["codebook"] for s in slices] == cbs
    assert np.array_equal(op.decode(buf), x)


def _pin_calibrated(op, fmt):
    from tests.test_payload import _per_slice_input
    x, cbs, escapes = _per_slice_input(fmt)
    buf = op.write_calibrated(x, fmt, 8, 208)
    _, slices = op.read(buf)
    assert [s["codebook"] for s in slices] == cbs
    assert [s["n_escapes"] for s in slices] == escapes


PINS = ([lambda op, n=n: _pin_fixture(op, n) for n in FIXTURES] + [_pin_per_slice_codebooks]
        + [lambda op, f=f: _pin_calibrated(op, f) for f in ("bf16", "e5m2")])


def test_pins_hold_for_the_real_payload_oracle():
    with open(SRC) as f:
        op = _variant(f.read())
    for pin in PINS:
        pin(op)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_payload_mutation_is_caught(name):
    old, new = MUTATIONS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation target for {name} not found"
    op = _variant(src.replace(old, new, 1))
    failures = 0
    for pin in PINS:
        try:
            pin(op)
        except Exception:
            failures += 1
    assert failures > 0, f"no pin caught mutation {name}"

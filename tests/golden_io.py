"""Reader for the hand-worked fixtures in tests/golden/."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            out[key] = rest.split()
    return out


def hex_array(tokens, dtype):
    return np.array([int(t, 16) for t in tokens], dtype=dtype)


def int_array(tokens, dtype):
    return np.array([int(t) for t in tokens], dtype=dtype)


def fixture_streams(fx: dict) -> dict:
    fmt = fx["format"][0]
    return {
        "fmt": fmt,
        "chunk": int(fx["chunk"][0]),
        "codebook": int_array(fx["codebook"], np.uint8),
        "input": hex_array(fx["input_hex"], np.uint16 if fmt == "bf16" else np.uint8),
        "codes": hex_array(fx["codes_hex"], np.uint8),
        "signman": hex_array(fx["signman_hex"], np.uint8),
        "esc_pos": int_array(fx["esc_pos"], np.uint16),
        "esc_val": int_array(fx["esc_val"], np.uint8),
        "chunk_off": int_array(fx["chunk_off"], np.uint32),
        "compressed_bytes": int(fx["compressed_bytes"][0]),
    }


STREAM_FIXTURES = ["bf16_tiny_chunk8.txt", "bf16_tiny_chunk4.txt", "e5m2_tiny_chunk8.txt"]

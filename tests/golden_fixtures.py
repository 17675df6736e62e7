"""Parser for the hand-written golden fixtures under tests/golden/."""
import os
import re

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
_HEX = re.compile(r"^[0-9a-f]{2}$")


def _is_row(tokens):
    return len(tokens) > 0 and all(_HEX.match(t) for t in tokens)


def parse(name: str) -> dict:
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]
    out = {}
    key = None
    for ln in lines:
        tok = ln.split()
        if _is_row(tok) and key is not None and isinstance(out.get(key), list):
            out[key].append(bytes(int(t, 16) for t in tok))
            continue
        key = tok[0]
        rest = tok[1:]
        if not rest:
            out[key] = []  # a block of rows follows
        elif key in ("device_idx", "host_idx"):
            out[key] = np.array([int(t) for t in rest], dtype=np.int64)
        elif key in ("device_fill", "host_fill"):
            out[key] = rest[0]
        else:
            out[key] = int(rest[0])
    return out


def device_image(fx: dict):
    """Device layer images described by the fixture's device_fill."""
    L, R, S = fx["num_layers"], fx["row_bytes"], fx["device_slots"]
    fill = fx["device_fill"]
    layers = []
    for l in range(L):
        if fill.startswith("rule:"):
            spec = fill[len("rule:"):].split(",")
            rows = []
            for d in range(S):
                row = [l if s == "l" else d if s == "d" else int(s, 16) for s in spec]
                assert len(row) == R
                rows.append(row)
            layers.append(np.array(rows, dtype=np.uint8).reshape(-1))
        else:
            layers.append(np.full(S * R, int(fill, 16), dtype=np.uint8))
    return layers


def rows_image(rows) -> np.ndarray:
    return np.frombuffer(b"".join(rows), dtype=np.uint8).copy()

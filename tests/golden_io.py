"""Reader for the text fixtures under tests/golden/."""
import os

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

HAND_K2_SHAPES = {
    "h_history": (1, 2, 2), "h_s2": (1, 2), "W_A": (2, 1), "W_B": (2, 1), "W_C": (2, 1),
    "W_O": (1, 2), "d_h_enriched": (1, 2), "h_enriched": (1, 2),
    "d_h_history": (1, 2, 2), "d_h_s2": (1, 2), "dW_A": (2, 1), "dW_B": (2, 1),
    "dW_C": (2, 1), "dW_O": (1, 2),
}


def load(name: str, shapes: dict) -> dict:
    out = {}
    with open(os.path.join(GOLDEN_DIR, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            arr = np.array([float(v) for v in vals], dtype=np.float64)
            out[key] = float(arr[0]) if key == "tw" else arr.reshape(shapes[key])
    return out


def hand_k2() -> dict:
    return load("hand_k2.txt", HAND_K2_SHAPES)

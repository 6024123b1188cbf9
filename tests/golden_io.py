"""Reader for the text fixtures under tests/golden (key: row ; row ; ...)."""
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, val = line.split(":", 1)
            rows = [[float(v) for v in r.split()] for r in val.split(";")]
            arr = np.array(rows, dtype=np.float64)
            out[key.strip()] = arr[0] if len(rows) == 1 else arr
    return out

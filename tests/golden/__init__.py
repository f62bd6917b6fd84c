"""Readers for the text fixtures in this folder (values printed on the pages)."""
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))


def load(name: str) -> dict:
    """Parse `key: int int ...` lines; '#' starts a comment."""
    out = {}
    with open(os.path.join(_HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = np.array([int(x) for x in v.split()], dtype=np.int64)
    return out

"""Reader for the ``name = value  # citation`` fixture files in this folder."""
from __future__ import annotations

import os

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(HERE, name), encoding="utf-8") as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (p.strip() for p in line.split("=", 1))
            parts = val.split()
            vals = [float(p) for p in parts]
            out[key] = vals[0] if len(vals) == 1 else vals
    return out

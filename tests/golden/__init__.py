"""Parser for the text fixtures in this folder (``key = value`` lines)."""

import os

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name):
    """Return ``{key: str}`` from ``tests/golden/<name>``, comments dropped."""
    out = {}
    with open(os.path.join(HERE, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            out[key] = val
    return out


def ints(val):
    return [int(x) for x in val.split()]

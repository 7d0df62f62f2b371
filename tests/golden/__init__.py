"""Stored expected values, each copied from the pages with its citation."""
import os

_DIR = os.path.dirname(os.path.abspath(__file__))


def load(name: str) -> dict:
    """Parse a ``key = value`` fixture (``#`` lines are the citation)."""
    out = {}
    with open(os.path.join(_DIR, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (x.strip() for x in line.split("=", 1))
            out[k] = float(v)
    return out

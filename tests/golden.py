"""Reader for the small text fixtures under tests/golden/ (``key: values`` lines)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            out[key.strip()] = val.split()
    return out


def floats(v):
    return [float(t) for t in v]


def ints(v):
    return [int(t) for t in v]

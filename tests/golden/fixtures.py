"""Reader for the hand-worked text fixtures in this folder."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))


def read(name: str) -> dict:
    """Parse ``key: value`` lines, skipping ``#`` comments."""
    out = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, value = line.split(":", 1)
            out[key.strip()] = value.strip()
    return out


def ints(s: str):
    return [int(v, 0) for v in s.split()]


def hexbytes(s: str):
    return [int(v, 16) for v in s.split()]

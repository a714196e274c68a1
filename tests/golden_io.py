"""Reader for the text fixtures under tests/golden/ (no arithmetic)."""

import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_blocks(name):
    """Parse ``[NAME rows cols]`` blocks of whitespace-separated numbers."""
    blocks, cur, shape = {}, None, None
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                key, r, c = line.strip("[]").split()
                cur, shape = key, (int(r), int(c))
                blocks[cur] = []
                continue
            blocks[cur].append([float(v) for v in line.split()])
    return {k: np.array(v, dtype=np.float64).reshape(
        len(v), len(v[0])) for k, v in blocks.items()}


def read_rows(name):
    """Parse a whitespace table (comment lines skipped) into a list of rows."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows

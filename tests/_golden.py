"""Readers for the text fixtures under tests/golden/ (each file cites the
page passage its values come from)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def keyvals(name):
    """'key: value' lines -> dict of str -> str (comments skipped)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split(":", 1)
                out[k.strip()] = v.strip()
    return out


def table(name):
    """Whitespace-separated rows -> list of lists of str (comments skipped)."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def ints(s):
    return [int(v, 0) for v in s.split()]


def floats(s):
    return [float(v) for v in s.split()]

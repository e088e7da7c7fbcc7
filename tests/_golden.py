"""Readers for the text fixtures under tests/golden/ (each file cites its source)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            s = raw.strip()
            if s and not s.startswith("#"):
                yield s


def cases(name, body_lines):
    """Split a fixture into cases: 'case <name> [k=v ...]' then body_lines lines."""
    it = iter(list(lines(name)))
    out = []
    for head in it:
        parts = head.split()
        assert parts[0] == "case", head
        attrs = dict(p.split("=", 1) for p in parts[2:] if "=" in p)
        flags = [p for p in parts[2:] if "=" not in p]
        body = [next(it) for _ in range(body_lines)]
        out.append((parts[1], attrs, flags, body))
    return out

"""Readers for the hand-worked fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            s = raw.split("#", 1)[0].strip()
            if s:
                yield s.split()


def keyed(name):
    out = {}
    for parts in lines(name):
        out.setdefault(parts[0], []).append(parts[1:])
    return out

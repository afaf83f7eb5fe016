"""Readers for the hand-worked fixtures under tests/golden/."""
import math
import os

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(tok: str) -> float:
    tok = tok.strip()
    if tok in ("nan", "inf", "-inf"):
        return float(tok)
    neg = tok.startswith("-")
    body = tok[1:] if neg else tok
    if "*" in body:
        a, b = body.split("*")
        v = _num(a) * _num(b)
    elif body.startswith("p"):
        v = math.ldexp(1.0, int(body[1:]))
    else:
        v = float(body)
    return -v if neg else v


def _lines(name):
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [t.strip() for t in line.split("|")]


def hand_blocks():
    """Yields (name, values[32] floats, scale byte, codes[32])."""
    for name, fill, over, scale, cfill, cover in _lines("hand_blocks.txt"):
        vals = [_num(fill)] * 32
        if over != "-":
            for item in over.split(","):
                i, v = item.split(":")
                vals[int(i)] = _num(v)
        codes = [int(cfill, 16)] * 32
        if cover != "-":
            for item in cover.split(","):
                i, v = item.split(":")
                codes[int(i)] = int(v, 16)
        yield name, vals, int(scale), codes


def swiglu_hand():
    """Yields ('fwd', g, u, h) and ('bwd', dh, g, u, dgate, dup)."""
    for row in _lines("swiglu_hand.txt"):
        yield (row[0],) + tuple(float(t) for t in row[1:])

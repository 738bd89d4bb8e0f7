"""Parser for the small text fixtures in this folder (exact fractions, ';' row separators)."""
from __future__ import annotations

import os
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))


def _num(tok: str):
    if tok in ("-inf", "+inf", "inf"):
        return float(tok)
    return Fraction(tok)


def load(name: str) -> dict:
    out = {}
    with open(os.path.join(HERE, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            rows = [[_num(t) for t in r.split()] for r in val.split(";")]
            out[key] = rows if len(rows) > 1 else rows[0]
    return out

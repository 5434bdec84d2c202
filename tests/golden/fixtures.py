"""Reader for the hand-derived closed-form fixtures in this folder."""
import math
import os
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))


def _num(tok: str) -> float:
    if tok.startswith("ln"):
        return math.log(float(tok[2:]))
    if "/" in tok:
        return float(Fraction(tok))
    return float(tok)


def load(name: str) -> list[dict]:
    """Parse ``name``: blocks of "key: values" lines, '#' comments, a new case
    starting whenever a key repeats."""
    cases, cur = [], {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            key = key.strip()
            if key in cur:
                cases.append(cur)
                cur = {}
            cur[key] = [_num(t) for t in vals.split()]
    if cur:
        cases.append(cur)
    return cases

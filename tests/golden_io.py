"""Reader for the text fixtures under tests/golden/ (key = value lines, '#' comments)."""
import math
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _num(tok: str) -> float:
    if tok == "ln3":
        return math.log(3.0)
    return float(tok)


def read_kv(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or "=" not in line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            vals = [_num(t) for t in val.split()]
            out[key] = vals if len(vals) > 1 else vals[0]
    return out


def read_mask_pictures(name: str = "causal_mask_pictures.txt"):
    cases = []
    with open(os.path.join(GOLDEN, name)) as f:
        lines = [ln.split("#", 1)[0].strip() for ln in f]
    lines = [ln for ln in lines if ln]
    i = 0
    while i < len(lines):
        tag, sq, skv = lines[i].split()
        assert tag == "case"
        sq, skv = int(sq), int(skv)
        rows = [[int(c) for c in lines[i + 1 + r]] for r in range(sq)]
        cases.append((sq, skv, rows))
        i += 1 + sq
    return cases

"""Reader for the small text fixtures under tests/golden/ ('#' comments, 'key = values' lines,
or whitespace-separated rows)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_kv(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            vals = [float(v) if any(c in v for c in ".e") else int(v) for v in val.split()]
            out[key] = vals[0] if len(vals) == 1 else vals
    return out


def read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows

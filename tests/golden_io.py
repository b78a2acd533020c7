"""Reader for the text fixtures under tests/golden/ ("key: values" lines, matrix
blocks after a bare "key:" line, '#' comments)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name):
    out, key = {}, None
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                key = k.strip()
                v = v.strip()
                if v:
                    out[key] = [int(t, 0) for t in v.split()]
                    key = None
                else:
                    out[key] = []
                continue
            if key is not None:
                out[key].append([int(t, 0) for t in line.split()])
    return out


def load_counts(name):
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            rows.append(([int(t) for t in lhs.split()], int(rhs)))
    return rows

"""Reader for the small text fixtures in tests/golden (``key = v1, v2, ...`` lines, '#' comments)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load(name, raw=False):
    """Values per key as floats (raw=True: as the printed strings)."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            vals = [v.strip() for v in val.split(",")]
            out[key] = vals if raw else [float(v) for v in vals]
    return out


def half_unit(printed):
    """Half a unit in the last printed decimal of each string (the print's own rounding)."""
    out = []
    for s in printed:
        dec = len(s.split(".", 1)[1]) if "." in s else 0
        out.append(0.5 * 10.0 ** (-dec))
    return out

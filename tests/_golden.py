"""Reader of the text fixtures under tests/golden/: '#' lines are the
citation, every other line is 'key: value value ...'."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.split()
    return out

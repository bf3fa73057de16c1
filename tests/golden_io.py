"""Readers for the hand-derived fixtures under tests/golden/."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_fixture(name):
    """Parse 'key: values' lines and 'key:' blocks of rows; '#' starts a comment."""
    out, block = {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].rstrip()
            if not line.strip():
                continue
            if ":" in line and not line[0].isspace() and not line.split(":", 1)[1].strip():
                block = line.split(":", 1)[0].strip()
                out[block] = []
                continue
            if ":" in line and not line[0].isdigit() and not line[0] == "-":
                key, val = line.split(":", 1)
                key = key.strip()
                if key == "case":
                    out.setdefault("case", []).append(dict(kv.split("=") for kv in val.split()))
                else:
                    out[key] = val.split()
                block = None
                continue
            if block is not None:
                out[block].append(line.split())
    return out

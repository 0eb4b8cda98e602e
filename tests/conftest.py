import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def load_golden(name):
    """Parse a golden fixture: '#' comments; 'key v v | v v' lines ('|' separates rows).

    Values are ints (decimal or 0x hex), floats, 'i:v' pairs or words; each key maps to a
    list of rows, each row a list of values."""
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            rows = []
            for part in rest.split("|"):
                vals = []
                for tok in part.split():
                    if ":" in tok:
                        a, b = tok.split(":")
                        vals.append((int(a), float(b)))
                    elif tok.lower().startswith("0x"):
                        vals.append(int(tok, 16))
                    else:
                        try:
                            vals.append(int(tok))
                        except ValueError:
                            try:
                                vals.append(float(tok))
                            except ValueError:
                                vals.append(tok)
                rows.append(vals)
            out[key] = rows
    return out


@pytest.fixture
def golden():
    return load_golden

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU case")


def load_golden(path):
    """Parse tests/golden/*.txt blocks into dicts (see the file header for fields)."""
    cases = []
    cur = None
    with open(path) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                cur = {"name": rest}
                cases.append(cur)
            elif key == "x":
                cur["x"] = [float(t) for t in rest.split()]
            elif key == "k":
                cur["k"] = int(rest)
            elif key == "p":
                cur["p"] = float(rest)
            elif key == "kept":
                cur["kept"] = sorted(int(t) for t in rest.split())
            elif key == "status":
                cur["status"] = rest
            elif key == "ambiguous":
                cur["ambiguous"] = bool(int(rest))
            else:
                raise ValueError(f"bad golden line: {line}")
    return cases


# flagged top-p rows per workload, reported at the end of the run
_FLAGGED = {}


@pytest.fixture(scope="session")
def record_flagged():
    """record_flagged(name, flagged, rows): the oracle's count of top-p rows
    whose boundary mass lies within 1e-6 * p of p, for the run summary."""

    def rec(name, flagged, rows):
        _FLAGGED[name] = (int(flagged), int(rows))

    return rec


def pytest_terminal_summary(terminalreporter):
    if _FLAGGED:
        terminalreporter.write_line("rows compared with the oracle, and the flagged top-p rows among them:")
        for name in sorted(_FLAGGED):
            f, n = _FLAGGED[name]
            terminalreporter.write_line(f"  {name}: {n} rows, {f} flagged")


@pytest.fixture(scope="session")
def golden_rows():
    return load_golden(os.path.join(ROOT, "tests", "golden", "handworked_rows.txt"))

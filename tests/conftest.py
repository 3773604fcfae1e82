import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
for p in (ROOT, ROOT / "tests"):
    if str(p) not in sys.path:
        sys.path.insert(0, str(p))

# (label, {name: value}) records of the GPU parity tests: attention errors and
# near-tie counts against the oracle, printed after the run (also under -q).
_PARITY: list[tuple[str, dict]] = []


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


@pytest.fixture(scope="session")
def parity():
    """report(label, **numbers): one line of the parity summary."""
    def report(label, **kv):
        _PARITY.append((label, kv))
    return report


def _fmt(v):
    if isinstance(v, float):
        return f"{v:.3e}"
    return str(v)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    if not _PARITY:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity against the oracle (attention errors; ids: near-ties / hard mismatches)")
    for label, kv in _PARITY:
        tr.write_line(f"{label}: " + " ".join(f"{k}={_fmt(v)}" for k, v in kv.items()))

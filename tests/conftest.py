import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The randomised oracle properties need hypothesis, which not every machine
# has (the GPU hosts do not); leave the module out there instead of reporting
# a skip: its tests are CPU tests and run wherever hypothesis is installed.
try:
    import hypothesis  # noqa: F401
    collect_ignore = []
except ImportError:
    collect_ignore = ["test_oracle_properties.py"]


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter):
    """Threshold-boundary mask flips of every parity trajectory that ran: bits
    of the GPU's mask that differ from the oracle's, over the bits compared."""
    try:
        from tests._harness import REPORTS
    except Exception:
        return
    rows = [r for r in REPORTS if r.mask_bits]
    if not rows:
        return
    tr = terminalreporter
    tr.write_sep("-", "mask flips against the oracle (fraction of mask bits compared)")
    flips = sum(r.flips for r in rows)
    bits = sum(r.mask_bits for r in rows)
    worst = max(rows, key=lambda r: r.flip_fraction)
    tr.write_line(f"{len(rows)} trajectories, {bits} mask bits compared, {flips} flipped "
                  f"(fraction {flips / bits:.3g}); largest: {worst.flip_fraction:.3g} in "
                  f"{worst.name}")
    for r in rows:
        if "shards" in r.name:
            tr.write_line(f"  {r.name}: {r.flips} of {r.mask_bits} bits "
                          f"(fraction {r.flip_fraction:.3g}), bit-identical: {r.exact}")

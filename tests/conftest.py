import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter):
    """Error margins of the GPU parity checks: per mode, the largest element error as a
    fraction of its band, and every TF32 case (the loosest band) by name."""
    try:
        from gpu_helpers import MARGINS
    except Exception:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.section("parity margins (largest error / band)")
    for mode in ("bf16", "fp32", "tf32"):
        got = [m for m in MARGINS if m[0] == mode]
        if got:
            w = max(got, key=lambda m: m[2])
            tr.write_line(f"{mode}: {len(got)} checks, worst {w[2]:.3f} ({w[1]})")
    for mode, what, worst in MARGINS:
        if mode == "tf32":
            tr.write_line(f"  tf32 {what}: {worst:.3f}")

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a library)")


def pytest_terminal_summary(terminalreporter):
    """List the error figures of every GPU-vs-oracle comparison made in the session."""
    harness = sys.modules.get("harness")
    records = getattr(harness, "RECORDS", None)
    if not records:
        return
    tr = terminalreporter
    tr.section("parity: max-abs / max-rel (vs max(|ref|, 1)) / LSE max-abs against the oracle")
    worst = [0.0, 0.0, 0.0]
    for test, n, max_abs, max_rel, lse in records:
        lse_s = f"{lse:.2e}" if lse is not None else "-"
        tr.write_line(f"{max_abs:.2e} {max_rel:.2e} {lse_s:>8}  {n:>9}  {test}")
        worst = [max(worst[0], max_abs), max(worst[1], max_rel), max(worst[2], lse or 0.0)]
    tr.write_line(f"worst over {len(records)} comparisons: max-abs {worst[0]:.3e}, max-rel {worst[1]:.3e}, "
                  f"LSE {worst[2]:.3e}")

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(scope="session", autouse=True)
def _built_libraries():
    """Compile the CUDA library and the oracle once per session (no-op when up to date)."""
    from attention_relative_position_gb300 import _build
    import oracle
    _build.build()
    oracle.build()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the max-abs error of every GPU-vs-oracle comparison made in this run (and write
    them as JSON to $FAT_PARITY_LOG when that is set)."""
    gc = sys.modules.get("gpu_common")
    log = getattr(gc, "PARITY_LOG", None) if gc is not None else None
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", f"parity: {len(log)} comparisons (max-abs error, GPU vs oracle)")
    tr.write_line(f"{'case':42s} {'output':6s} {'oracle':10s} {'max_abs':>9s} "
                  f"{'|ref|<4':>9s} {'max|ref|':>9s} {'err/tol':>7s} ok")
    for r in log:
        extra = f" rel {r['rel']:.2e}" if "rel" in r else ""
        tr.write_line(f"{r['case'][:42]:42s} {r['output']:6s} {r['mode']:10s} "
                      f"{r['max_abs']:9.2e} {r['max_abs_small']:9.2e} {r['max_ref']:9.2e} "
                      f"{r['worst_ratio']:7.3f} {'yes' if r['ok'] else 'NO'}{extra}")
    path = os.environ.get("FAT_PARITY_LOG")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(log, f, indent=0)

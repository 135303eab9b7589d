import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The largest attention error the parity checks saw, and the near-ties
    they counted (kind: ties of compared items), so a run's tail records
    both."""
    pu = sys.modules.get("parity_util")
    errs = getattr(pu, "ERR_MAX", None) if pu is not None else None
    if errs and errs["attention rel"] > 0:
        terminalreporter.write_line(
            f"largest attention error vs the oracle: row-relative {errs['attention rel']:.3e} "
            f"(tolerance {pu.ATTN_RTOL:g}), lse absolute {errs['lse abs']:.3e}")
    counts = getattr(pu, "TIE_COUNTS", None) if pu is not None else None
    if not counts:
        return
    parts = [f"{k}: {v[1]} of {v[0]}" for k, v in sorted(counts.items())]
    terminalreporter.write_line("near-ties counted (tie band 1e-5): " + "; ".join(parts))

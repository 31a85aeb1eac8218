import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running oracle comparison")


def pytest_terminal_summary(terminalreporter):
    """Raw max-abs errors of the comparisons made in this session, grouped by output name, against
    the flat bounds; FA_PARITY_LOG=<path> also writes every record as JSON."""
    import json
    try:
        from helpers import ERROR_LOG
    except ImportError:
        return
    if not ERROR_LOG:
        return
    groups = {}
    for r in ERROR_LOG:
        key = (r["what"].split()[0] if r["what"] else "?", r["flat_bound"], r["rel"] > 0)
        g = groups.setdefault(key, {"n": 0, "worst": 0.0, "worst_ref": 0.0, "held": 0})
        g["n"] += 1
        g["held"] += r["flat_bound_held"]
        if r["max_abs_err"] >= g["worst"]:
            g["worst"], g["worst_ref"] = r["max_abs_err"], r["max_abs_ref"]
    terminalreporter.write_sep("-", "parity: raw max |err| against the flat bound")
    for (name, bound, rel), g in sorted(groups.items()):
        terminalreporter.write_line(
            f"{name:<24} checks {g['n']:4d}  worst |err| {g['worst']:.3e} (|ref| up to {g['worst_ref']:.3g})  "
            f"flat bound {bound:.0e}{' + 2^-8|ref|' if rel else ''}: flat bound alone held in {g['held']}/{g['n']}")
    path = os.environ.get("FA_PARITY_LOG")
    if path:
        with open(path, "w") as f:
            json.dump(ERROR_LOG, f, indent=0)

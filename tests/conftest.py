import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """One line per layer parity comparison of the session: rel-L2 (bar 5e-3),
    max-abs/rms beyond the output's bf16 rounding (bar 2e-2) and the literal
    max-abs/rms beside it, near-tie tokens, tokens whose ids differ."""
    try:
        from _common import PARITY_LOG
    except ImportError:
        return
    if not PARITY_LOG:
        return
    tr = terminalreporter
    tr.write_sep("-", "layer parity vs the fp64 oracle")
    tr.write_line(f"{'case':58s} {'rel-L2':>9s} {'max/rms':>9s} {'literal':>9s} near mism")
    for r in PARITY_LOG:
        tr.write_line(f"{r['name'][:58]:58s} {r['rel']:9.2e} {r['max']:9.2e} {r['literal']:9.2e} "
                      f"{r.get('near', '-'):>4} {r.get('mism', '-'):>4}")

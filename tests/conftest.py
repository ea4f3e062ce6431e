import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU check")


def pytest_terminal_summary(terminalreporter):
    """One line per output comparison with the oracle: elements compared, the
    largest bf16 difference and how many bf16 elements passed only through the
    one-bf16-step allowance (differences above 1.5e-2 on values whose bf16 step
    is larger)."""
    tl = sys.modules.get("gk_testlib")
    rows = getattr(tl, "REPORT", None) if tl else None
    if not rows:
        return
    tw = terminalreporter
    tw.section("outputs against the oracle")
    for what, st in rows:
        line = (f"{what or '(unnamed)'}: {st['elements']} elements, bf16 max {st['bf16_max']:.3g}, "
                f"{st['bf16_widened']} within one bf16 step only")
        if "f32_max" in st:
            line += f", f32 max {st['f32_max']:.3g}"
        tw.write_line(line)

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Parity margins of every GPU-vs-oracle comparison of the session."""
    try:
        from helpers import MARGINS
    except ImportError:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.section("parity margins (GPU vs oracle)")
    for m in MARGINS:
        if "code_mismatch_rate" in m:
            tr.write_line(f"{m['what']}: mismatch {m['code_mismatch_rate']:.2e} of {m['n']} codes, "
                          f"non-adjacent {m['non_adjacent']}")
        else:
            extra = (f"  | vs bf16(ref) rel_l2 {m['rel_l2_vs_bf16_ref']:.2e}, flips {m['bf16_flips']:.2%}"
                     if "rel_l2_vs_bf16_ref" in m else "")
            tr.write_line(f"{m['what']}: rel_l2 {m['rel_l2']:.2e}  max_abs {m['max_abs']:.2e}{extra}")

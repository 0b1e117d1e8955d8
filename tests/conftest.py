import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large-size parity case")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Excused mask blocks of every GPU-vs-oracle mask comparison of the run: a block whose
    GPU and oracle bits differ is excused only when its oracle score lies within 1e-4
    relative of the row's threshold, its radius within 1e-4 of the median, or its row holds
    an excused centroid-path block.  Unexcused mismatches fail the test that met them."""
    try:
        from parity_util import EXCUSE_LOG
    except Exception:
        return
    if not EXCUSE_LOG:
        return
    tr = terminalreporter
    tr.write_sep("-", "excused mask blocks (GPU vs oracle)")
    by_test = {}
    for test, label, compared, excused in EXCUSE_LOG:
        by_test.setdefault(test, []).append((label, compared, excused))
    for test, recs in by_test.items():
        c = sum(r[1] for r in recs)
        e = sum(r[2] for r in recs)
        line = f"{test}: {e} excused of {c} compared"
        labelled = [r for r in recs if r[0]]
        if len(labelled) > 1:
            line += " | " + " ".join(f"{lab}={exc}" for lab, _, exc in labelled)
        tr.write_line(line)
    tot_c = sum(r[2] for r in EXCUSE_LOG)
    tot_e = sum(r[3] for r in EXCUSE_LOG)
    tr.write_line(f"all mask comparisons: {tot_e} excused blocks of {tot_c} compared "
                  f"({len(EXCUSE_LOG)} comparisons, 0 unexcused)")

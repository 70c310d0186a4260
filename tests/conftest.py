import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """The parity margins of the run: every checked error against its
    tolerance (the closest cases first), so the log shows how much of each
    bound the kernels use."""
    gpu_util = sys.modules.get("gpu_util")
    margins = getattr(gpu_util, "MARGINS", None)
    if not margins:
        return
    rows = sorted(margins, key=lambda m: -m[2] / m[3])
    tr = terminalreporter
    tr.write_sep("-", "parity margins (max rel err / tolerance), %d checks" % len(rows))
    for test, name, err, tol in rows[:12]:
        tr.write_line("%5.3f  %.3e / %.0e  %-3s %s" % (err / tol, err, tol, name, test))
    worst = {}
    for test, name, err, tol in rows:
        if "training" in test:
            worst[name] = max(worst.get(name, 0.0), err)
    if worst:
        tr.write_line("training workload (bf16, sampled): " +
                      ", ".join("%s %.3e" % (k, v) for k, v in sorted(worst.items())))

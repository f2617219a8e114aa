import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large sampled-row parity cases")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print every parity check's literal figures against the exact oracle: the
    number of elements, the relative Frobenius error, max |got - exact|, how many
    elements exceed the absolute bound, the largest per-row allowance delta taken
    from the oracle's stored-precision result, in how many rows that allowance
    exceeds the absolute bound (rows where the oracle's own bf16-storage result
    misses it), and the worst excess over the element bound (<= 0 passes). The layer
    outputs of the five workloads come last."""
    gu = sys.modules.get("gpu_util")
    recs = [r for r in getattr(gu, "RECORDS", []) if not r[0].startswith("checker:")]
    if not recs:
        return
    tr = terminalreporter
    tr.section("parity against the oracle")
    tr.write_line(f"{'check':<44} {'elements':>9} {'rel_fro':>8} {'max|err|':>9} "
                  f"{'>atol':>6} {'atol':>8} {'delta':>8} {'d>atol':>9} {'excess':>9}")
    line = lambda r: (f"{r[0][:44]:<44} {r[1]:>9} {r[2]:>8.2e} {r[3]:>9.3e} {r[4]:>6} "
                      f"{r[5]:>8.2e} {r[6]:>8.2e} {f'{r[9]}/{r[8]}':>9} {r[7]:>+9.2e}")
    key = ("tiny out", "small out", "7b-16k out rows", "7b-64k out rows", "7b-128k out rows")
    for r in recs:
        if r[0] not in key:
            tr.write_line(line(r))
    last = [r for k in key for r in recs if r[0] == k]
    if last:
        tr.write_line("layer outputs of the five workloads (max|err| against the exact oracle):")
        for r in last:
            tr.write_line(line(r))

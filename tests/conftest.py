import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built extension")
    config.addinivalue_line("markers", "slow: long CPU runs")


def pytest_sessionfinish(session, exitstatus):
    """Writes the parity errors the GPU tests observed (per comparison: max and mean |diff|
    and the largest per-(row, head) ratio to the scaled bound) to $PA_PARITY_STATS."""
    path = os.environ.get("PA_PARITY_STATS")
    mod = sys.modules.get("tests.gpu_util")
    if not path or mod is None:
        return
    import json
    with open(path, "w") as f:
        json.dump([{"what": w, "max_abs": a, "mean_abs": m, "max_scaled": r}
                   for w, a, m, r in mod.STATS], f, indent=1)

import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    oracle.build()
    return oracle


def _parity_log():
    mod = sys.modules.get("_parity")
    return list(getattr(mod, "LOG", [])) if mod is not None else []


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Report every GPU-vs-oracle comparison of the session: compared units
    and evaluated tiles, tiles whose oracle vote statistic lies within the
    near-margin band of ln(lambda), and the decisions that differ there (the
    only place they may differ).  SSATTN_PARITY_REPORT=<path> also writes the
    records as JSON."""
    log = _parity_log()
    if not log:
        return
    tr = terminalreporter
    tr.section("parity against the oracle (near-margin decisions reported)")
    by_test = {}
    for r in log:
        t = by_test.setdefault(r.test or "?", dict(checks=0, units=0, tiles=0, skipped=0, near=0,
                                                     disagree=0, max_abs=0.0, max_abs_gpu_mask=0.0))
        t["checks"] += 1
        for key in ("units", "tiles", "skipped", "near", "disagree"):
            t[key] += getattr(r, key)
        t["max_abs"] = max(t["max_abs"], r.max_abs)
        t["max_abs_gpu_mask"] = max(t["max_abs_gpu_mask"], r.max_abs_gpu_mask)
    for name, t in by_test.items():
        if t["near"] or t["disagree"]:
            tr.write_line(f"{name}: {t['tiles']} tiles, {t['near']} near-margin, "
                          f"{t['disagree']} decisions differ (near-margin), "
                          f"max-abs {t['max_abs']:.2e}")
    tot = {k: sum(t[k] for t in by_test.values()) for k in ("checks", "units", "tiles", "skipped",
                                                             "near", "disagree")}
    worst = max(t["max_abs"] for t in by_test.values())
    worst_g = max(t["max_abs_gpu_mask"] for t in by_test.values())
    tr.write_line(f"total: {tot['checks']} launches checked, {tot['units']} units, "
                  f"{tot['tiles']} evaluated tiles ({tot['skipped']} skipped), "
                  f"{tot['near']} near-margin tiles, {tot['disagree']} decisions differ "
                  f"(all near-margin); output max-abs {worst:.2e} (own decisions), "
                  f"{worst_g:.2e} (under the GPU's decisions)")
    path = os.environ.get("SSATTN_PARITY_REPORT")
    if path:
        os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
        with open(path, "w") as f:
            json.dump({"totals": tot, "max_abs": worst, "max_abs_gpu_mask": worst_g,
                       "by_test": by_test,
                       "records": [r.__dict__ for r in log]}, f, indent=1, default=float)

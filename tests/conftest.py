import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    gh = sys.modules.get("gpu_helpers")
    if gh is not None:
        gh.close_oracle_pool()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the parity figures the bf16 checks recorded: the max-norm relative error
    (the asserted bound) and the elementwise relative error with a 1e-3 max|ref| floor."""
    gh = sys.modules.get("gpu_helpers")
    rows = getattr(gh, "PARITY", None) if gh is not None else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("bf16 parity against the fp64 oracle")
    tr.write_line(f"{'check':58s} {'tensor':14s} {'elements':>11s} {'max-norm':>9s} "
                  f"{'elem max':>9s} {'elem p99':>9s}")
    for label, tensor, n, e, emax, e99 in rows:
        tr.write_line(f"{label[:58]:58s} {tensor[:14]:14s} {n:11d} {e:9.2e} {emax:9.2e} "
                      f"{e99:9.2e}")
    path = os.environ.get("KDA_PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump([dict(zip(("check", "tensor", "elements", "maxnorm_rel", "elem_rel_max",
                                 "elem_rel_p99"), r)) for r in rows], f, indent=1)

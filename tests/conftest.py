import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libsk.so")
    config.addinivalue_line("markers", "slow: long-running GPU parity case")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped only on a machine without any CUDA device. On a GPU
    # machine a missing or unloadable library is a failure, never a skip.
    try:
        import torch

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this machine")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    # Strict-form GEMM parity: per labelled case, how many outputs lay more
    # than one BF16 ulp from the oracle's correctly rounded result (accepted
    # only through the cancellation bound).
    try:
        from parity import GEMM_RECORDS
    except ImportError:  # pragma: no cover
        return
    if not GEMM_RECORDS:
        return
    tr = terminalreporter
    tr.write_sep("-", "GEMM outputs beyond 1 BF16 ulp of the oracle (strict form)")
    total = sum(r[1] for r in GEMM_RECORDS)
    outs = sum(r[2] for r in GEMM_RECORDS)
    for label, n_ii, n, dmax in GEMM_RECORDS:
        tr.write_line(f"{label}: {n_ii} of {n} beyond 1 ulp (max distance {dmax} ulp)")
    tr.write_line(f"all cases: {total} of {outs} outputs beyond 1 ulp ({total / max(outs, 1):.2e})")


def read_cases(name):
    """Parse a golden fixture: ``key: values`` lines, cases split by blank lines."""
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if line.startswith("#"):
                continue
            if not line:
                if cur:
                    cases.append(cur)
                    cur = {}
                continue
            key, _, val = line.partition(":")
            cur[key.strip()] = val.split()
    if cur:
        cases.append(cur)
    return cases


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle

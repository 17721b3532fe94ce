import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity case (runs the oracle for many seconds)")


def pytest_terminal_summary(terminalreporter):
    """Score parity totals: how many compared scores the floored rule and the
    pure relative rule (no floor) each reject."""
    try:
        from parity import REPORT
    except ImportError:
        return
    if not REPORT:
        return
    n = sum(r[1] for r in REPORT)
    floored = sum(r[2] for r in REPORT)
    pure = sum(r[3] for r in REPORT)
    terminalreporter.write_line(
        f"score parity: {len(REPORT)} comparisons, {n} scores; outside the floored rule: {floored}; "
        f"outside the pure relative rule (no floor): {pure}")
    worst = sorted((r for r in REPORT if r[3]), key=lambda r: -r[3])[:5]
    for what, cnt, fl, pu in worst:
        terminalreporter.write_line(f"  {what}: {pu} of {cnt} scores outside the pure relative rule")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def _ensure_library():
    """Builds the CUDA library in-tree when it is missing (nvcc cross-compiles
    without a GPU); the binding itself never falls back to anything else."""
    so = os.path.join(ROOT, "shared_latent_key_cache_b300", "libli_b300.so")
    if not os.path.exists(so):
        import importlib.util
        path = os.path.join(ROOT, "shared_latent_key_cache_b300", "_build.py")
        spec = importlib.util.spec_from_file_location("li_b300_build", path)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()


@pytest.fixture(scope="session")
def li():
    """The CUDA library's Python binding (fails loudly when it cannot load)."""
    _ensure_library()
    import shared_latent_key_cache_b300 as m
    return m

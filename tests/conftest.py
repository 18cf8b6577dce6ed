import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.hookimpl(tryfirst=True)
def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running case")
    # temporary files (the mutated oracle builds) stay inside the repository's
    # ignored build folder, one directory per session, removed at its end
    if config.option.basetemp is None:
        config.option.basetemp = os.path.join(ROOT, "tests", "_build", f"pytest-{os.getpid()}")
        config._dg_own_basetemp = config.option.basetemp


def pytest_unconfigure(config):
    own = getattr(config, "_dg_own_basetemp", None)
    if own:
        import shutil
        shutil.rmtree(own, ignore_errors=True)


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle

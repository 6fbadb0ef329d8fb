import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture
def tune(monkeypatch):
    """Sets TPGEMM_* planner overrides for one test. The library reads them
    once into a snapshot, so every change is followed by a reload; at the end
    the environment is restored and read again."""
    import tile_primitive_tensor_gb300 as tp

    class Tune:
        def setenv(self, name, value):
            monkeypatch.setenv(name, value)
            tp.tpgemm_reload_tuning()

        def delenv(self, name):
            monkeypatch.delenv(name)
            tp.tpgemm_reload_tuning()

    yield Tune()
    monkeypatch.undo()
    tp.tpgemm_reload_tuning()

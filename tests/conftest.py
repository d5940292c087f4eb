import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


import pytest  # noqa: E402


@pytest.fixture
def hooks(monkeypatch):
    """Sets or clears the library's SSM_* test-hook environment variables for one test.
    The library reads them once, so every change is followed by a reload, and the
    original environment is restored (and reloaded) when the test ends."""
    import selective_state_space_154_b300 as ssm

    class Hooks:
        def set(self, name, value):
            monkeypatch.setenv(name, str(value))
            ssm.reload_test_hooks()

        def unset(self, name):
            monkeypatch.delenv(name, raising=False)
            ssm.reload_test_hooks()

    yield Hooks()
    monkeypatch.undo()
    ssm.reload_test_hooks()

"""The entry point's smoke run (one small call of every step, checked against
the oracle) as part of the GPU suite, so a change that breaks it shows up
with the other GPU tests."""
import pytest

pytestmark = pytest.mark.gpu


def test_graft_entry_smoke_runs():
    import __graft_entry__
    __graft_entry__.smoke()

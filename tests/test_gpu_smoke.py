"""The round-end smoke check (one small call against the oracle) runs in the
GPU suite as well, so that a change to the binding or the library that breaks
it shows up here."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_entry_point():
    import __graft_entry__ as g
    g.smoke()

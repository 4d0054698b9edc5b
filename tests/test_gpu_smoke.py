"""The smoke entry point (one small step + one gather on cuda:0, checked
against the oracle) keeps working."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_entry_point(zlib):
    import __graft_entry__
    __graft_entry__.smoke()

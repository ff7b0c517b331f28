"""The entry point's smoke() runs as it does before a benchmark: one small
DEFERRED verify/commit sequence checked against the oracle."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_entry_point(gdn):
    import __graft_entry__
    __graft_entry__.smoke()

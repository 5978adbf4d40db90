"""__graft_entry__.smoke(): the one small layer forward checked against the
oracle on cuda:0."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_runs_and_passes():
    import __graft_entry__ as g
    g.smoke()

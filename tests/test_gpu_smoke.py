"""__graft_entry__.smoke() -- the small end-to-end check run on a fresh GPU
box -- passes: layout, FP8 dispatch, the one-call layout + dispatch and the
rank-grouped combine against the oracle."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_passes(capsys):
    import __graft_entry__
    __graft_entry__.smoke()
    assert "smoke ok" in capsys.readouterr().out

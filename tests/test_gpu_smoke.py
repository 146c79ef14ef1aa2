"""The entry point's smoke check runs as it will at a GPU machine's start."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_entry_point(capsys):
    import __graft_entry__

    __graft_entry__.smoke()
    assert "smoke ok" in capsys.readouterr().out

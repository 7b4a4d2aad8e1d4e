"""The entry point's smoke() (one small Muon step over a wide, a tall and a
packed tensor plus one AdamW step, each checked against the oracle) passes."""
import pytest

pytestmark = pytest.mark.gpu


def test_smoke_passes():
    import __graft_entry__
    __graft_entry__.smoke()

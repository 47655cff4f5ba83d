"""The package entry's one-shot check (a tiny group: forward, loss, backward, finalize on
cuda:0, compared with the oracle) runs clean."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.gpu
def test_smoke_entry_point_passes():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import __graft_entry__ as entry
    entry.smoke()

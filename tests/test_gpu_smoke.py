"""The round-trip check of __graft_entry__.smoke() runs as a test too: one
tiny forward + backward through the C ABI on cuda:0, compared with the oracle
(planner arrays bit-exact, O/LSE/dQ/dK/dV within the stated tolerances),
plus the materialisation gather and the raw-order sum."""
import os
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_smoke_entry_point():
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import __graft_entry__
    __graft_entry__.smoke()

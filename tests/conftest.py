import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: a long CPU-oracle case")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


class attn_schedule:
    """Context manager: runs the block with the attention schedule of the
    default handle set to (kernel, max_ctas, min_tiles, splits)
    (tt_set_attn_schedule), then restores the default."""

    def __init__(self, tt, kernel: int, max_ctas: int = 0, min_tiles: int = 0, splits: int = 0):
        self.tt, self.args = tt, (kernel, max_ctas, min_tiles, splits)

    def __enter__(self):
        self.tt.handle().set_attn_schedule(*self.args)
        return self

    def __exit__(self, *exc):
        self.tt.handle().set_attn_schedule(0, 0, 0, 0)
        return False


# (kernel, max_ctas, min_tiles, splits): the schedule chosen by shape; the
# persistent kernel with query tiles cut between CTAs in different ways (one
# CTA, a few, pieces of one tile); one unit per CTA with forced KV splits.
SCHEDULES = [(0, 0, 0, 0), (2, 1, 1, 0), (2, 2, 1, 0), (2, 3, 1, 0), (2, 7, 1, 0), (2, 0, 1, 0),
             (2, 0, 0, 0), (1, 0, 0, 1), (1, 0, 0, 2), (1, 0, 0, 3), (1, 0, 0, 7)]
# both kernels at their defaults
KERNELS = [(1, 0, 0, 0), (2, 0, 0, 0)]

"""Scale relayout bit-exactness, the bounded-wait failure path, and launch counting."""
import numpy as np
import pytest
import torch

import block_scaled_precision_mma_gb300 as bs
import oracle
from tests.gpu_common import to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    bs.build()
    bs.load()
    torch.cuda.init()


@pytest.mark.parametrize("role", ["A", "B"])
@pytest.mark.parametrize("rows,kblocks", [(1, 1), (128, 4), (300, 11), (8192, 256),
                                          (14336, 448), (129, 9), (4096, 128)])
def test_relayout_bit_exact(rows, kblocks, role):
    s = np.random.default_rng([3, rows, kblocks]).integers(0, 255, size=(rows, kblocks),
                                                           dtype=np.uint8)
    got = bs.mx_scale_relayout(to_dev(s), role).cpu().numpy()
    assert np.array_equal(got, oracle.wide_scale_relayout(s, bs.ROLES[role]))


def test_wait_timeout_is_reported_and_context_survives():
    """A wait on a barrier nothing completes gives up after its limit and latches
    BSMMA_DEV_TIMEOUT; the context keeps working afterwards."""
    assert bs.probe_wait_timeout(50_000_000) == 6
    assert bs.device_status() == 0
    x = torch.ones(1024, device="cuda")
    assert float(x.sum().item()) == 1024.0


def test_launch_count_increments():
    n0 = bs.launch_count()
    s = torch.zeros((256, 8), dtype=torch.uint8, device="cuda")
    bs.mx_scale_relayout(s, "A")
    torch.cuda.synchronize()
    assert bs.launch_count() == n0 + 1

"""The parity recorder's device-side measure (used where an output is too
large to copy to the host) computes the oracle's normwise and elementwise
errors exactly, over a tensor split into pieces (CPU tensors here)."""
import numpy as np
import torch

from oracle import moe_ref as ref
from tests import parity_log


def test_device_measures_equal_the_oracle_definitions():
    rng = np.random.default_rng(3)
    for shape in ((300, 7), (40, 3, 5), (1, 1)):
        want = rng.standard_normal(shape) * 3.0
        want.flat[::7] = 0.0                     # elements below the floor
        got = want + rng.standard_normal(shape) * 1e-3
        g, w = torch.from_numpy(got), torch.from_numpy(want)
        cut = max(1, shape[0] // 3)
        nw, ew = parity_log.assert_close_device(
            [(g[:cut], w[:cut]), (g[cut:], w[cut:])], 1.0, "pieces")
        assert nw == ref.normwise_error(got, want)
        assert ew == ref.elementwise_error(got, want)
    z = np.zeros((4, 4))
    d = z + 0.5
    nw, ew = parity_log.assert_close_device(
        [(torch.from_numpy(d), torch.from_numpy(z))], 1.0, "zero reference")
    assert nw == ref.normwise_error(d, z) and ew == ref.elementwise_error(d, z)
    parity_log.RECORDS.clear()

"""The oracle against its committed regression record (tests/golden/)."""
import os

import numpy as np

from tests.golden.make_golden import compute

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_fp32_forward_matches_record():
    rows = [l for l in open(os.path.join(HERE, "golden", "tiny_fp32_fwd.txt"))
            if not l.startswith("#")]
    vals = [np.array([float(v) for v in l.split()]) for l in rows]
    y_rec, h_rec = np.stack(vals[:16]), np.stack(vals[16:])
    y, hL = compute()
    np.testing.assert_allclose(y[0], y_rec, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(hL[0], h_rec, rtol=1e-13, atol=1e-15)

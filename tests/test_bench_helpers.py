"""Host-side helpers of bench.py (CPU): the fidelity measures against the oracle's."""
import numpy as np
import torch

import bench
import oracle as O


def test_fidelity_stats_match_the_oracle():
    rng = np.random.default_rng(31)
    g = rng.standard_normal((40, 70)).astype(np.float32)
    g_hat = (g + 0.01 * rng.standard_normal(g.shape)).astype(np.float32)
    got = bench.fidelity_stats(torch.from_numpy(g_hat), torch.from_numpy(g).double())
    want = O.fidelity(g_hat, g)
    for key in ("rel_l2", "cos", "max_err", "mse"):
        assert np.isclose(got[key], want[key], rtol=1e-12, atol=0), key
    exact = bench.fidelity_stats(torch.from_numpy(g), torch.from_numpy(g))
    assert exact["rel_l2"] == 0 and exact["max_err"] == 0 and np.isclose(exact["cos"], 1)


def test_fidelity_stats_are_strict_json():
    zero = torch.zeros(3, 4)
    got = bench.fidelity_stats(zero, torch.ones(3, 4))
    assert got["cos"] is None and got["rel_l2"] == 1.0

"""The FLOP counts bench.py reports, against brute force on small shapes (CPU)."""
import numpy as np
import pytest

import bench
from attention_backward_flashattention_gb300 import synthetic as syn


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("density", [0.1, 0.5, 1.0])
def test_block_sparse_pairs_match_brute_force(causal, density):
    """visible_pairs counts the (query, key) pairs that the kept blocks and the
    causal band leave, the quantity the block-sparse TFLOP/s divide by."""
    w = syn.Workload("acct", 2, 3, 512, 64, 64, causal)
    mask = bench.block_sparse_mask(w, density, seed=7)
    assert mask.shape == (1, 3, 4, 4)
    assert np.all(mask[0, :, np.arange(4), np.arange(4)] == 1)  # diagonal kept
    i = np.arange(w.T)[:, None]
    j = np.arange(w.T)[None, :]
    band = (j <= i) if causal else np.ones((w.T, w.T), bool)
    count = 0
    for h in range(w.H):
        keep = np.kron(mask[0, h], np.ones((128, 128), np.uint8)).astype(bool)
        count += int((keep & band).sum())
    assert bench.visible_pairs(w, mask) == w.B * count


def test_dense_flops_match_the_formula():
    """With every block kept the pair count gives the workload's FLOP formula
    (2*B*H*T^2*(3*dqk + 2*dv), halved for causal up to the diagonal's T/2)."""
    for causal in (False, True):
        w = syn.Workload("acct", 1, 2, 1024, 128, 128, causal)
        mask = np.ones((1, w.H, 8, 8), np.uint8)
        pairs = bench.visible_pairs(w, mask)
        exact = w.B * w.H * (w.T * (w.T + 1) // 2 if causal else w.T * w.T)
        assert pairs == exact
        flops = 2.0 * pairs * (3 * w.dqk + 2 * w.dv)
        assert abs(flops - w.bwd_flops()) <= (2.0 * w.B * w.H * w.T / 2 * (3 * w.dqk + 2 * w.dv)
                                              if causal else 0.0)

"""The seeded synthetic inputs follow their stated recipe: the configurations'
shapes and recipes, bf16 values, the same draws for the same seed, and the
value distributions and structure (N(0,1) activations, N(0,0.02) weights,
Laplace(0,1) for the [1,32] prefill, round(0.001 K) outlier channels x50 for
the [1,128] prefill)."""
import math

import numpy as np
import pytest
import torch

from fp8_block_scaled_sgq_gb300 import synth


def test_configuration_shapes_and_recipes():
    w = synth.WORKLOADS
    assert [(c.M, c.N, c.K, c.blk_n, c.blk_k, c.ue8m0) for c in w["tiny"]] == [(16, 256, 512, 128, 128, False)]
    assert [c.M for c in w["decode_block32"]] == [1, 4, 16, 64]
    assert {(c.N, c.K, c.blk_n, c.blk_k, c.ue8m0) for c in w["decode_block32"]} == {(7168, 2048, 32, 32, True)}
    p128, = w["prefill_block128"]
    assert (p128.M, p128.N, p128.K, p128.blk_n, p128.blk_k, p128.ue8m0) == (4096, 7168, 7168, 128, 128, True)
    assert p128.outlier_frac == 0.001 and p128.dist == "normal"
    p32, = w["prefill_block32"]
    assert (p32.M, p32.N, p32.K, p32.blk_n, p32.blk_k, p32.ue8m0, p32.dist) == (4096, 4096, 7168, 32, 32, True,
                                                                                 "laplace")
    sweep = {(c.M, c.N, c.K, c.blk_k) for c in w["sweep"]}
    assert sweep == {(m, n, k, b) for m in (1, 2, 4, 8, 32, 128, 512, 2048, 8192)
                     for (n, k) in ((24576, 1536), (1536, 7168)) for b in (128, 32)}
    assert all(c.group == c.blk_k for cs in w.values() for c in cs)


def test_bf16_and_seeded():
    a = synth.activation(8, 256, seed=3)
    assert a.dtype == torch.bfloat16 and a.shape == (8, 256)
    assert torch.equal(a, synth.activation(8, 256, seed=3))
    assert not torch.equal(a, synth.activation(8, 256, seed=4))
    w = synth.weight(16, 256, seed=3)
    assert w.dtype == torch.bfloat16 and torch.equal(w, synth.weight(16, 256, seed=3))
    # weights draw with seed + 1, so they are not the activations' draws
    assert not torch.equal(synth.weight(8, 256, seed=3).float() / 0.02, a.float())


def test_value_distributions():
    x = synth.activation(512, 2048, seed=1).float().numpy()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    w = synth.weight(512, 2048, seed=1).float().numpy()
    assert abs(w.mean()) < 2e-4 and abs(w.std() - 0.02) < 2e-4
    lap = synth.activation(512, 2048, seed=1, dist="laplace").float().numpy()
    # Laplace(0, 1): mean 0, mean |x| = 1, variance 2, excess kurtosis 3
    assert abs(lap.mean()) < 0.01 and abs(np.abs(lap).mean() - 1.0) < 0.01
    assert abs(lap.var() - 2.0) < 0.05
    kurt = ((lap - lap.mean()) ** 4).mean() / lap.var() ** 2 - 3.0
    assert abs(kurt - 3.0) < 0.3


@pytest.mark.parametrize("K", [2048, 7168])
def test_outlier_channels(K):
    """round(0.001 K) whole channels (columns) scaled by 50; the rest N(0, 1)."""
    M = 256
    x = synth.activation(M, K, seed=0, outlier_frac=0.001).float().numpy()
    col_std = x.std(axis=0)
    n_out = int(round(0.001 * K))
    big = np.nonzero(col_std > 10.0)[0]
    assert len(big) == n_out
    assert np.all(np.abs(col_std[big] / 50.0 - 1.0) < 0.2)
    rest = np.delete(x, big, axis=1)
    assert abs(rest.std() - 1.0) < 0.02
    base = synth.activation(M, K, seed=0).float().numpy()
    # the same draws, scaled (bf16 rounding aside) in exactly those channels
    np.testing.assert_array_equal(np.delete(base, big, axis=1), rest)
    assert math.isclose(float(np.abs(x[:, big]).mean() / np.abs(base[:, big]).mean()), 50.0, rel_tol=0.01)

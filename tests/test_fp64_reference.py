"""The GPU-side fp64 reference of the full-D parity tests (test_full_d_gpu.py),
run on the CPU against the oracle on small shapes of both recipes, ragged N:
the same definition (dequantise, then an fp64 product) in two codes must agree
to fp64 rounding, for D and for the bound Sum_k |a||w|."""
import numpy as np
import pytest
import torch

from fp8_block_scaled_sgq_gb300 import synth

import oracle
from test_full_d_gpu import fp64_reference


@pytest.mark.parametrize("M,N,K,bn,bk", [(70, 300, 512, 128, 128), (33, 264, 256, 32, 32), (5, 136, 384, 128, 32)])
@pytest.mark.parametrize("ue8m0", [True, False])
def test_fp64_reference_matches_the_oracle(M, N, K, bn, bk, ue8m0):
    c = synth.Case("ref", M, N, K, bn, bk, ue8m0, seed=M + N)
    aq, a_s = oracle.quant_token_group(c.x(), bk, ue8m0)
    wq, ws = oracle.quant_weight_block(c.w(), bn, bk, ue8m0)
    t = [torch.from_numpy(np.ascontiguousarray(v)) for v in (aq, a_s, wq, ws)]
    ref, bound = fp64_reference(*t, bn, bk)
    d, b = oracle.gemm(aq, a_s, wq, ws, bn, bk)
    assert np.abs(ref.numpy() - d).max() <= 1e-12 * b.max()
    assert np.abs(bound.numpy() - b).max() <= 1e-12 * b.max()


@pytest.mark.parametrize("M,N,K", [(7, 264, 512), (70, 136, 2048)])
@pytest.mark.parametrize("per_row", [True, False])
def test_scaled_mm_reference_matches_the_oracle(M, N, K, per_row):
    from test_full_d_gpu import scaled_mm_reference
    aq, sa = oracle.quant_per_token(synth.activation(M, K, seed=M))
    wq, sb = oracle.quant_per_token(synth.weight(N, K, seed=N))
    if not per_row:
        sa = np.array([np.float32(0.0113)], dtype=np.float32)
    bias = synth.activation(1, N, seed=3).reshape(N)
    t = [torch.from_numpy(np.ascontiguousarray(v)) for v in (aq, sa, wq, sb)]
    ref, bound = scaled_mm_reference(*t, bias)
    d, b = oracle.scaled_mm(aq, sa, wq, sb, bias)
    assert np.abs(ref.numpy() - d).max() <= 1e-12 * (b.max() + 1.0)
    assert np.abs(bound.numpy() - b).max() <= 1e-12 * b.max()

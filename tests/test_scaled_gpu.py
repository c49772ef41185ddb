"""Per-token and per-tensor FP8 quantisation and fp8_scaled_mm on the GPU
against the CPU oracle ("Sgl project Sglang GEMM Interface": the
sgl_per_token_quant_fp8 / sgl_per_tensor_quant_fp8 routines and
fp8_scaled_mm).  Codes and scales bit-exact; D within the GEMM tolerance
(D read as fp64; the bound carries the scales)."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import synth

import oracle
from common import check_gemm, tile_rows

pytestmark = pytest.mark.gpu


def edge_rows(x):
    x = x.clone()
    if x.shape[0] > 3:
        x[1] = 0.0
        x[2, : x.shape[1] // 2] = -0.0
        x[3, 5] = 6.0e4
    return x


@pytest.mark.parametrize("M,K", [(1, 16), (7, 2048), (33, 7168), (300, 1056), (4096, 7168)])
def test_per_token_bit_exact(M, K):
    x = edge_rows(synth.activation(M, K, seed=M + K))
    q, s = sgq.quant_per_token(x.cuda())
    assert sgq.sgq_device_status() == 0
    oq, os_ = oracle.quant_per_token(x)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("shape", [(16,), (3, 48), (64, 2048), (4096, 7168)])
@pytest.mark.parametrize("static", [False, True])
def test_per_tensor_bit_exact(shape, static):
    n = int(np.prod(shape))
    x = synth.activation(1, n, seed=n).reshape(shape)
    if n > 64:
        x.view(-1)[7] = 5.0e3
    scale = 0.0172 if static else None
    q, s = sgq.quant_per_tensor(x.cuda(), scale)
    assert sgq.sgq_device_status() == 0
    oq, os_ = oracle.quant_per_tensor(x, scale)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert s.cpu().numpy()[0] == os_[0]


def _operands(M, N, K, seed):
    x = synth.activation(M, K, seed=seed)
    w = synth.weight(N, K, seed=seed + 1)
    aq, sa = oracle.quant_per_token(x)
    wq, sb = oracle.quant_per_token(w)        # per-output-channel weight scales
    return aq, sa, wq, sb


@pytest.mark.parametrize("M,N,K", [(1, 264, 2048), (16, 7168, 2048), (64, 1032, 2080), (200, 520, 1024),
                                   (1000, 1032, 4096)])
@pytest.mark.parametrize("mode", ["row_col_bias", "tensor_tensor", "row_tensor", "tensor_col_bias"])
def test_scaled_mm_vs_oracle(M, N, K, mode):
    aq, sa, wq, sb = _operands(M, N, K, seed=M + N)
    if "tensor_tensor" in mode or mode.startswith("tensor"):
        sa = np.array([np.float32(0.0113)], dtype=np.float32)
    if mode.endswith("tensor") and not mode.startswith("row_col"):
        sb = np.array([np.float32(0.00071)], dtype=np.float32)
    bias = synth.activation(1, N, seed=N).reshape(N) if "bias" in mode else None
    d = sgq.fp8_scaled_mm(torch.from_numpy(aq).cuda(), torch.from_numpy(sa).cuda(), torch.from_numpy(wq).cuda(),
                          torch.from_numpy(sb).cuda(), None if bias is None else bias.cuda())
    assert sgq.sgq_device_status() == 0
    rows = np.arange(M) if M <= 200 else tile_rows(M, seed=M)
    sa_r = sa if sa.size == 1 else sa[rows]
    dref, bound = oracle.scaled_mm(aq[rows], sa_r, wq, sb, bias)
    check_gemm(d[torch.from_numpy(rows).cuda()], dref, bound, f"scaled_mm M={M} N={N} K={K} {mode}")


def test_scaled_mm_prefill_every_tile():
    """Full prefill size (4096 x 7168 x 7168), per-row x per-column scales and
    bias: one row of every 64-row block compared over all N columns."""
    M, N, K = 4096, 7168, 7168
    aq, sa, wq, sb = _operands(M, N, K, seed=9)
    bias = synth.activation(1, N, seed=N).reshape(N)
    d = sgq.fp8_scaled_mm(torch.from_numpy(aq).cuda(), torch.from_numpy(sa).cuda(), torch.from_numpy(wq).cuda(),
                          torch.from_numpy(sb).cuda(), bias.cuda())
    assert sgq.sgq_device_status() == 0
    rows = tile_rows(M, seed=9)
    dref, bound = oracle.scaled_mm(aq[rows], sa[rows], wq, sb, bias)
    check_gemm(d[torch.from_numpy(rows).cuda()], dref, bound, "scaled_mm prefill")


def test_scaled_mm_split_k_deterministic_and_end_to_end():
    """Per-token quantisation feeding fp8_scaled_mm on one stream; split-K
    (decode-sized M) sums in a fixed order."""
    M, N, K = 16, 7168, 2048
    x = synth.activation(M, K, seed=3)
    w = synth.weight(N, K, seed=4)
    wq, sb = sgq.quant_per_token(w.cuda())
    aq, sa = sgq.quant_per_token(x.cuda())
    d0 = sgq.fp8_scaled_mm(aq, sa, wq, sb)
    for _ in range(3):
        assert torch.equal(d0, sgq.fp8_scaled_mm(aq, sa, wq, sb))
    oaq, osa = oracle.quant_per_token(x)
    owq, osb = oracle.quant_per_token(w)
    dref, bound = oracle.scaled_mm(oaq, osa, owq, osb)
    check_gemm(d0, dref, bound, "per-token quant -> scaled_mm")

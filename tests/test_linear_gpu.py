"""Quantise-and-multiply (sgq_fp8_block_linear) on the GPU.

At decode-sized M it is one kernel whose epilogue warps quantise the bf16
activation tiles into shared memory.  Its codes and scales must equal the
stand-alone quantisation kernel's (and the oracle's) bit for bit, and its D
must equal the two-call path's (quantisation kernel, then the GEMM) bit for
bit, since the MMAs see the same operands in the same order.  D is also
checked against the oracle under the GEMM tolerance."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq
from fp8_block_scaled_sgq_gb300 import binding, synth

import oracle
from common import check_gemm

pytestmark = pytest.mark.gpu

RECIPES = [(32, 32), (128, 128), (128, 32), (32, 128)]


def two_call(x, wq, ws, bn, bk, ue):
    xq, xs = sgq.quant_token_group(x, bk, ue)
    d = sgq.fp8_block_gemm(xq, xs, wq, ws, bn, bk)
    return d, xq, xs


def fused(x, wq, ws, bn, bk, ue, outputs=True):
    M, K = x.shape
    d = torch.empty((M, wq.shape[0]), dtype=torch.bfloat16, device="cuda")
    xq = torch.full((M, K), 0x5A, dtype=torch.uint8, device="cuda") if outputs else None
    xs = torch.full((M, K // bk), -1.0, dtype=torch.float32, device="cuda") if outputs else None
    sgq.sgq_fp8_block_linear(x, int(ue), wq, ws, d, M, wq.shape[0], K, bn, bk, xq, xs)
    assert sgq.sgq_device_status() == 0
    return d, xq, xs


def make(M, N, K, bn, bk, ue, seed):
    x = synth.activation(M, K, seed=seed)
    w = synth.weight(N, K, seed=seed + 1)
    wq, ws = oracle.quant_weight_block(w, bn, bk, ue)
    return x, wq, ws


@pytest.mark.parametrize("M", [1, 4, 16, 32, 33, 64])
@pytest.mark.parametrize("bn,bk", RECIPES)
@pytest.mark.parametrize("ue", [True, False])
def test_fused_matches_two_calls_and_oracle(M, bn, bk, ue):
    N, K = 264, 2048
    x, wq, ws = make(M, N, K, bn, bk, ue, seed=M * 7 + bk)
    xd = x.cuda()
    wqd, wsd = torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda()
    d2, xq2, xs2 = two_call(xd, wqd, wsd, bn, bk, ue)
    d1, xq1, xs1 = fused(xd, wqd, wsd, bn, bk, ue)
    assert torch.equal(xq1, xq2)
    assert torch.equal(xs1, xs2)
    assert torch.equal(d1, d2)
    # without the xq/xs outputs every M <= 64 runs as one kernel
    d0, _, _ = fused(xd, wqd, wsd, bn, bk, ue, outputs=False)
    assert torch.equal(d0, d2)
    aq, a_s = oracle.quant_token_group(x, bk, ue)
    assert np.array_equal(xq1.cpu().numpy(), aq)
    assert np.array_equal(xs1.cpu().numpy(), a_s)
    dref, bound = oracle.gemm(aq, a_s, wq, ws, bn, bk)
    check_gemm(d1, dref, bound, f"fused M={M} blk=({bn},{bk}) ue8m0={ue}")


@pytest.mark.parametrize("idx", range(4))
def test_fused_decode_block32_full_size(idx):
    """The decode workload's shapes (N=7168, K=2048, [32,32], UE8M0): one
    kernel, D bit-identical to the two-call path, without the xq/xs outputs."""
    c = synth.WORKLOADS["decode_block32"][idx]
    x = c.x().cuda()
    w = c.w().cuda()
    wq, ws = sgq.quant_weight_block(w, c.blk_n, c.blk_k, True)
    d2, _, _ = two_call(x, wq, ws, c.blk_n, c.blk_k, True)
    before = sgq.sgq_launch_count()
    d1, _, _ = fused(x, wq, ws, c.blk_n, c.blk_k, True, outputs=False)
    assert sgq.sgq_launch_count() - before == 1
    assert torch.equal(d1, d2)


def test_fused_edge_values():
    """Zero groups (eps scale, zero codes), values that saturate nothing but sit
    at the E4M3 range, negative zeros, and a huge outlier channel."""
    M, N, K, bn, bk = 16, 136, 1024, 32, 32
    x = synth.activation(M, K, seed=21)
    x[3, :] = 0.0
    x[5, 64:96] = -0.0
    x[7, 10] = 3.0e4
    x[9, :] = torch.tensor(448.0, dtype=torch.bfloat16)
    for ue in (True, False):
        w = synth.weight(N, K, seed=22)
        wq, ws = oracle.quant_weight_block(w, bn, bk, ue)
        wqd, wsd = torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda()
        d2, xq2, xs2 = two_call(x.cuda(), wqd, wsd, bn, bk, ue)
        d1, xq1, xs1 = fused(x.cuda(), wqd, wsd, bn, bk, ue)
        assert torch.equal(xq1, xq2) and torch.equal(xs1, xs2) and torch.equal(d1, d2)
        d0, _, _ = fused(x.cuda(), wqd, wsd, bn, bk, ue, outputs=False)   # one kernel
        assert torch.equal(d0, d2)
        aq, a_s = oracle.quant_token_group(x, bk, ue)
        assert np.array_equal(xq1.cpu().numpy(), aq) and np.array_equal(xs1.cpu().numpy(), a_s)


def test_two_kernel_shapes_need_scratch():
    """Shapes that cannot be fused (M > 64, or K/blk_k not a multiple of 4) run
    the two kernels when xq/xs are given, and are refused without them."""
    for M, K in ((100, 1024), (8, 1056)):
        N, bn, bk = 264, 32, 32
        x, wq, ws = make(M, N, K, bn, bk, True, seed=M)
        xd = x.cuda()
        wqd, wsd = torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda()
        d = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        rc = binding.load_library().sgq_fp8_block_linear(xd.data_ptr(), 1, wqd.data_ptr(), wsd.data_ptr(),
                                                         d.data_ptr(), M, N, K, bn, bk, None, None, None)
        assert rc == binding.SGQ_ERR_UNSUPPORTED
        d2, _, _ = two_call(xd, wqd, wsd, bn, bk, True)
        d1, xq1, xs1 = fused(xd, wqd, wsd, bn, bk, True)
        assert torch.equal(d1, d2)
        aq, a_s = oracle.quant_token_group(x, bk, True)
        assert np.array_equal(xq1.cpu().numpy(), aq)


def test_fused_split_k_deterministic():
    x, wq, ws = make(16, 7168, 2048, 32, 32, True, seed=5)
    xd = x.cuda()
    wqd, wsd = torch.from_numpy(wq).cuda(), torch.from_numpy(ws).cuda()
    d0, _, _ = fused(xd, wqd, wsd, 32, 32, True, outputs=False)
    for _ in range(3):
        d1, _, _ = fused(xd, wqd, wsd, 32, 32, True, outputs=False)
        assert torch.equal(d0, d1)

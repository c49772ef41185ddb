"""V2 per-token-group quantisation on the GPU (fused SiLU-and-mul, masked M)
against the CPU oracle: codes and scales bit-exact ("Sgl project Sglang GEMM
Interface", Quantization Routines: the V2 variant of
sgl_per_token_group_quant_8bit).  The fused path's exp is a published method
implemented on both sides; it is also checked against CUDA's own expf."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_sgq_gb300 as sgq

import oracle

pytestmark = pytest.mark.gpu


def v2_input(E, T, W, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn((E, T, W), generator=g) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("E,T,H", [(1, 1, 32), (1, 7, 2048), (4, 33, 7168), (8, 64, 1536)])
@pytest.mark.parametrize("group,ue", [(32, True), (128, False), (128, True)])
@pytest.mark.parametrize("fuse", [False, True])
def test_v2_bit_exact(E, T, H, group, ue, fuse):
    if H % group:
        pytest.skip("H must hold whole groups")
    x = v2_input(E, T, 2 * H if fuse else H, seed=E * T + H, scale=4.0)
    q, s = sgq.quant_token_group_v2(x.cuda(), group, ue, fuse)
    assert sgq.sgq_device_status() == 0
    oq, os_ = oracle.quant_token_group_v2(x, group, ue, fuse)
    assert np.array_equal(q.cpu().numpy(), oq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))


def test_v2_masked_rows_untouched_and_edges():
    E, T, H = 4, 9, 256
    x = v2_input(E, T, 2 * H, seed=5, scale=20.0)      # gates beyond the exp range and around 0
    x[0, 0, :H] = 0.0
    x[1, 2, :8] = 120.0
    x[1, 2, 8:16] = -120.0
    masked = torch.tensor([0, 9, 3, 12], dtype=torch.int32)   # 12 > T: all rows
    xq = torch.full((E, T, H), 0x5A, dtype=torch.uint8, device="cuda")
    xs = torch.full((E, T, H // 32), -1.0, dtype=torch.float32, device="cuda")
    sgq.quant_token_group_v2(x.cuda(), 32, True, True, masked.cuda(), xq, xs)
    assert sgq.sgq_device_status() == 0
    oq, os_ = oracle.quant_token_group_v2(x, 32, True, True, masked.numpy(),
                                           xq=np.full((E, T, H), 0x5A, np.uint8),
                                           xs=np.full((E, T, H // 32), -1.0, np.float32))
    assert np.array_equal(xq.cpu().numpy(), oq)
    assert np.array_equal(xs.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert (xq[0].cpu().numpy() == 0x5A).all() and (xq[2, 3:].cpu().numpy() == 0x5A).all()


def test_exp_against_cuda_expf():
    """The textbook exp (oracle implementation) stays within 2 ulp of CUDA's
    expf over the range the fused path uses; the kernel runs the same steps,
    which the bit-exact tests above confirm through the codes."""
    xs = torch.linspace(-87.0, 88.5, 200001, dtype=torch.float32)
    cuda_e = torch.exp(xs.cuda()).cpu().numpy()
    ours = oracle.exp_tc(xs.numpy())
    diff = np.abs(ours.view(np.int32).astype(np.int64) - cuda_e.view(np.int32).astype(np.int64))
    assert diff.max() <= 2

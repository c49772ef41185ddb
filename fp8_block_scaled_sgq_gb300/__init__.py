"""GB300 (sm_103a) W8A8 FP8 block-scaled linear layer.

The compute lives in ``libsgq.so`` (hand-written CUDA behind the C ABI of
``include/sgq.h``).  This package holds the ctypes binding (``binding``), the
nvcc build (``build``), seeded synthetic inputs (``synth``) and a few
torch-facing helpers below that only allocate outputs and call the binding.
"""
from __future__ import annotations

from .binding import (  # noqa: F401
    EXPORTS, SGQ_GEMM_DEFAULT, SGQ_GEMM_FORCE_PROMOTE, SGQ_GEMM_ISSUE_ALT, SGQ_GEMM_ISSUE_SINGLE, SgqError,
    SGQ_GEMM_SCALES_POW2, SGQ_GEMM_TEST_TIMEOUT,
    load_library, sgq_device_status,
    sgq_fp8_block_gemm, sgq_fp8_block_gemm_ex, sgq_fp8_block_linear, sgq_fp8_scaled_mm,
    sgq_quant_per_tensor, sgq_quant_per_token, sgq_quant_token_group_v2, sgq_launch_count, sgq_quant_token_group,
    sgq_allocated_bytes, sgq_fp8_block_gemm_ue8m0, sgq_quant_token_group_ue8m0, sgq_scales_to_ue8m0,
    sgq_gemm_plan, sgq_gemm_plan_pow2,
    sgq_quant_weight_block, sgq_version, status_string)


def quant_token_group(x, group: int, ue8m0: bool, stream=None):
    """bf16 [M, K] CUDA tensor -> (uint8 E4M3 codes [M, K], fp32 scales [M, K/group])."""
    import torch
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    xs = torch.empty((M, K // group), dtype=torch.float32, device=x.device)
    sgq_quant_token_group(x, M, K, group, ue8m0, xq, xs, stream)
    return xq, xs


def quant_weight_block(w, blk_n: int, blk_k: int, ue8m0: bool, stream=None):
    """bf16 [N, K] CUDA tensor -> (uint8 E4M3 [N, K], fp32 [ceil(N/blk_n), K/blk_k])."""
    import torch
    N, K = w.shape
    wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    ws = torch.empty(((N + blk_n - 1) // blk_n, K // blk_k), dtype=torch.float32, device=w.device)
    sgq_quant_weight_block(w, N, K, blk_n, blk_k, ue8m0, wq, ws, stream)
    return wq, ws


def fp8_block_gemm(aq, a_s, wq, ws, blk_n: int, blk_k: int, out=None, flags: int = 0, stream=None):
    """D = (Aq*As)(Wq*Ws)^T as a bf16 [M, N] CUDA tensor."""
    import torch
    M, K = aq.shape
    N = wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    sgq_fp8_block_gemm_ex(aq, a_s, wq, ws, out, M, N, K, blk_n, blk_k, flags, stream)
    return out


def quant_token_group_ue8m0(x, group: int, stream=None):
    """bf16 [M, K] CUDA tensor -> (uint8 E4M3 codes [M, K], UE8M0 scale bytes [M, K/group])."""
    import torch
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    xe = torch.empty((M, K // group), dtype=torch.uint8, device=x.device)
    sgq_quant_token_group_ue8m0(x, M, K, group, xq, xe, stream)
    return xq, xe


def scales_to_ue8m0(s, stream=None):
    """fp32 power-of-two scales (CUDA tensor) -> UE8M0 bytes of the same shape."""
    import torch
    s = s.contiguous()
    e = torch.empty(s.shape, dtype=torch.uint8, device=s.device)
    sgq_scales_to_ue8m0(s, s.numel(), e, stream)
    return e


def fp8_block_gemm_ue8m0(aq, ae, wq, we, blk_n: int, blk_k: int, out=None, flags: int = 0, stream=None):
    """D = (Aq*2^(Ae-127))(Wq*2^(We-127))^T as a bf16 [M, N] CUDA tensor."""
    import torch
    M, K = aq.shape
    N = wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    sgq_fp8_block_gemm_ue8m0(aq, ae, wq, we, out, M, N, K, blk_n, blk_k, flags, stream)
    return out


def w8a8_linear(x, wq, ws, blk_n: int, blk_k: int, ue8m0: bool, out=None, stream=None):
    """Quantise x per token group of blk_k, then the block-scaled GEMM (two calls)."""
    xq, xs = quant_token_group(x, blk_k, ue8m0, stream)
    return fp8_block_gemm(xq, xs, wq, ws, blk_n, blk_k, out=out, stream=stream)


def fp8_block_linear(x, wq, ws, blk_n: int, blk_k: int, ue8m0: bool, out=None, xq=None, xs=None, stream=None):
    """The same result as w8a8_linear through sgq_fp8_block_linear: one kernel
    at decode-sized M (xq/xs optional outputs), else two (xq/xs allocated here
    as scratch when not given)."""
    import torch
    M, K = x.shape
    N = wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    try:
        sgq_fp8_block_linear(x, ue8m0, wq, ws, out, M, N, K, blk_n, blk_k, xq, xs, stream)
    except SgqError as e:
        if e.status != 2 or xq is not None:   # SGQ_ERR_UNSUPPORTED: needs scratch
            raise
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
        xs = torch.empty((M, K // blk_k), dtype=torch.float32, device=x.device)
        sgq_fp8_block_linear(x, ue8m0, wq, ws, out, M, N, K, blk_n, blk_k, xq, xs, stream)
    return out


def quant_per_token(x, stream=None):
    """bf16 [M, K] CUDA tensor -> (E4M3 codes [M, K], fp32 scales [M])."""
    import torch
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    xs = torch.empty((M,), dtype=torch.float32, device=x.device)
    sgq_quant_per_token(x, M, K, xq, xs, stream)
    return xq, xs


def quant_per_tensor(x, scale=None, stream=None):
    """bf16 CUDA tensor -> (E4M3 codes, fp32 scale [1]); scale=None: dynamic."""
    import torch
    xq = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    xs = torch.empty((4,), dtype=torch.float32, device=x.device)   # 16-byte aligned; [0] is the scale
    if scale is not None:
        xs[0] = float(scale)
    sgq_quant_per_tensor(x, x.numel(), scale is not None, xq, xs, stream)
    return xq, xs[:1]


def fp8_scaled_mm(aq, sa, wq, sb, bias=None, out=None, stream=None):
    """D = bf16((Aq Wq^T) * sa * sb + bias): sa of 1 or M values, sb of 1 or N."""
    import torch
    M, K = aq.shape
    N = wq.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=aq.device)
    sgq_fp8_scaled_mm(aq, sa, sa.numel(), wq, sb, sb.numel(), bias, out, M, N, K, stream)
    return out


def quant_token_group_v2(x, group: int, ue8m0: bool, fuse: bool, masked_m=None, xq=None, xs=None, stream=None):
    """bf16 [E, T, W] CUDA tensor (W = 2H fused) -> (E4M3 [E, T, H], fp32 [E, T, H/group])."""
    import torch
    E, T, W = x.shape
    H = W // 2 if fuse else W
    if xq is None:
        xq = torch.empty((E, T, H), dtype=torch.uint8, device=x.device)
    if xs is None:
        xs = torch.empty((E, T, H // group), dtype=torch.float32, device=x.device)
    sgq_quant_token_group_v2(x, E, T, H, group, ue8m0, fuse, masked_m, xq, xs, stream)
    return xq, xs
